// Internal interfaces between the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace swg {

// Partial-sum layout shared by every split-K producer and the reduction:
//   part[((s * M + m) * 2 + gu) * d_ff + j]   (f32)
// s = K slice, m = row of x, gu = 0 for x.W_gate, 1 for x.W_up, j = column.
inline size_t partial_elems(int64_t slices, int64_t M, int64_t d_ff) {
  return (size_t)slices * (size_t)M * 2u * (size_t)d_ff;
}

struct SimtPlan {
  int vec;          // elements per 16-byte load (4 f32, 8 bf16)
  int cols_per_cta; // 32 lanes x vec
  int row_chunk;    // rows of x per CTA (1, 2 or 4)
  int64_t col_blocks, row_chunks, slices, k_per_slice;
  bool fused;       // single launch: the last slice of a column block reduces
  size_t counters_bytes;   // arrival counters of the single launch
  int cluster = 0;  // > 0: the cluster form (simt_cluster.cu) with this many K slices
};

// Tuning overrides from the environment (SWIGLU_SK_NB, SWIGLU_SK_PROMO,
// SWIGLU_SK_HINT, SWIGLU_SK_PREFETCH_UNITS, SWIGLU_SK_CLUSTER, SWIGLU_SK_BULK,
// SWIGLU_SK_SPLIT, SWIGLU_SK_KB, SWIGLU_TILE_PAIR, SWIGLU_TILE_SK, SWIGLU_TILE_SK_SPLIT,
// SWIGLU_TILE_SEQ, SWIGLU_TILE_BAND, SWIGLU_SIMT_FUSED, SWIGLU_SIMT_CLUSTER,
// SWIGLU_INJECT_OOM), read in one pass over the environment for every planned
// call, so a process may change them between calls.  -1: not set (the
// measured default applies).
struct Tuning {
  int sk_nb = -1, sk_promo = -1, sk_hint = -1, sk_prefetch_units = -1, sk_cluster = -1;
  int tile_pair = -1, tile_sk = -1, tile_sk_split = -1, tile_seq = -1, tile_band = -1;
  int simt_fused = -1;
  int sk_bulk = -1;   // skinny stream-K final sums staged by bulk copies (default on)
  int sk_kb = -1;     // skinny FP8: 64-deep k blocks per unit (1 or 2)
  int sk_split = -1;  // skinny stream-K final sums in a second kernel (1) or by the
                      // group's last CTA (0)
  int simt_cluster = -1;   // 0: never use the cluster form of the SIMT path;
                           // 4..8: that many K slices per cluster
  // Test hook (SWIGLU_INJECT_OOM=1): every workspace the library would take
  // from its pool or its per-stream cache fails to allocate, so the call
  // returns SWIGLU_ERR_OOM having enqueued nothing.  Caller workspaces and
  // calls that need none are unaffected.
  int inject_oom = 0;
};
Tuning read_tuning();

SimtPlan plan_simt(int64_t M, int64_t d, int64_t d_ff, int dtype, int num_sms,
                   const Tuning& tn = Tuning{});

// S1 (SIMT): partial sums of x.Wg and x.Wu per K slice.  With `counters`
// (p.fused plans; zero on entry unless !counters_clean, left at zero) the
// same launch also reduces them and writes h: no S2 launch follows.
// `packed`: wg (= wu) is a packed weight matrix (kWeightsPacked).
cudaError_t launch_simt_partial(const void* x, const void* wg, const void* wu,
                                float* part, int64_t M, int64_t d, int64_t d_ff,
                                int dtype, const SimtPlan& p, cudaStream_t st,
                                unsigned* counters = nullptr, bool counters_clean = false,
                                void* h = nullptr, bool packed = false);

// The cluster form of the SIMT path (M = 1, weights <= 32 MB, d <= 2048):
// the K slices of a column block are one thread-block cluster that adds them
// in distributed shared memory, in one launch with no workspace.  Returns the
// cluster size (the K slices, 4 ... 8) for a call it serves, else 0.
// caps[S] (S = 4 ... 8): clusters of S CTAs of its 4-CTAs-per-SM form that
// fit at once (simt_cluster_caps), or null to assume that 8-CTA clusters fit.
constexpr int kSimtCapSlots = 9;
int simt_cluster_plan(int64_t M, int64_t d, int64_t d_ff, int dtype, const Tuning& tn,
                      const int* caps = nullptr);
cudaError_t simt_cluster_caps(int caps[kSimtCapSlots]);
// Largest d for which AUTO prefers the cluster form for bf16 (at most 4 rows
// of W per thread, so 4 CTAs fit per SM).
constexpr int64_t kSimtClusterPreferMaxK = 1024;
cudaError_t launch_simt_cluster(const void* x, const void* wg, const void* wu, void* h,
                                int64_t M, int64_t d, int64_t d_ff, int dtype, int ks,
                                bool packed, cudaStream_t st);

// How the weights are stored:
//   kWeightsKN      [K, n_out] row-major (the default);
//   kWeightsNK      [n_out, K], K contiguous (torch.nn.Linear.weight);
//   kWeightsPacked  one [K, packed_cols(n_out)] matrix for W_gate and W_up
//                   (up projection only), see launch_pack.
enum WeightLayout : int { kWeightsKN = 0, kWeightsNK = 1, kWeightsPacked = 2 };

// Step a0: packed weights [d, packed_cols(d_ff)], 64-column blocks of W_gate
// and W_up alternating (zero past d_ff).  A packed matrix is read by the
// up-projection kernels with gate block b at packed column 128 b and up
// block b at 128 b + 64.
int64_t packed_cols(int64_t d_ff);
cudaError_t launch_pack(const void* wg, const void* wu, void* out, int64_t d, int64_t d_ff,
                        int dtype, int num_sms, cudaStream_t st);

// S2: fixed-order sum over slices, then h = silu(g) * u rounded to dtype.
cudaError_t launch_reduce_swiglu(const float* part, void* h, int64_t M,
                                 int64_t d_ff, int64_t slices, int dtype,
                                 int num_sms, cudaStream_t st);

// Entry-point checks shared by the C-ABI functions (defined in swiglu_api.cu):
// argument validation, the current device (sm_103 check and SM count), and
// the calling thread's error string.  Each returns a swiglu_status.
int api_validate(const void* x, const void* wg, const void* wu, const void* h, int64_t M,
                 int64_t d, int64_t d_ff, int dtype);
int api_current_device(int* dev, int* num_sms);
int api_fail(int status, const char* detail);
int api_cuda_fail(cudaError_t e, const char* what);
void api_clear_error();
unsigned* api_status_word(int dev);   // device address of the error word
constexpr int64_t kSimtMaxGridYZ = 65535;

// TMA descriptor of a row-major bf16 matrix [rows, cols], 128-byte swizzle.
cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                              int box_cols, int box_rows, int l2_promo_bytes = 256);

// Skinny tensor-core path (bf16, small M): swap-AB split-K over a balanced
// partition of (64-column block, 64-deep k block) units.
struct SkinnyPlan {
  int n_pad;               // M rounded up to the MMA N granule (16..256)
  int nb;                  // 64-column blocks per unit (1, 2 or 4)
  int kb;                  // 64-deep k blocks per unit (1, or 2 for FP8)
  int l2_promo;            // L2 promotion of the weight loads (bytes, 0 = none)
  int hint;                // weight-load L2 hint: 0 none, 1 evict_first
  bool plain;              // plain epilogue (down projection) instead of SwiGLU
  int prefetch_units;      // units each CTA prefetches into L2 before its dependency wait
  int cluster;             // cluster mode: CTAs per column group (0: stream-K)
  int bulk;                // stream-K: stage the final sums by bulk copies when possible
  int split;               // stream-K: the kernel only writes partial sums; a second
                           // kernel (launched with programmatic serialisation) adds them
  int64_t n_cb, n_kb;      // units: (nb x 64)-column groups, 64-deep k blocks
  int64_t units;           // n_cb * n_kb
  int grid;                // CTAs (<= SM count)
  int maxq;                // partial slots per column block
  size_t counters_bytes;   // arrival counters (zeroed before every launch)
  size_t part_bytes;       // partial sums
};
constexpr int kSkinnyMaxN = 256;
// Weights up to this size (bytes of the matrices one call streams) run the
// skinny kernel in cluster mode, larger ones in stream-K mode.
constexpr int64_t kSkinnyClusterMaxWeightBytes = (int64_t)32 << 20;
// Whether a down projection's 128-column groups fit as 4-CTA clusters all at
// once (cluster_caps: clusters of 2 / 4 / 8 skinny CTAs that fit, or null to
// assume 0.95 num_sms / 4 of them).
bool skinny_plain_cluster4_fits(int64_t K, int64_t n_out, int num_sms, const int* cluster_caps);
// K: shared dimension; n_out: output columns; plain: down-projection mode.
// cluster_caps[lg]: thread-block clusters of 2^lg CTAs of the skinny kernel
// that fit on the device at once (lg = 1..3), or null (an estimate from num_sms).
SkinnyPlan plan_skinny(int64_t M, int64_t K, int64_t n_out, int num_sms, bool plain,
                       bool fp8 = false, const int* cluster_caps = nullptr,
                       const Tuning& tn = Tuning{});
cudaError_t skinny_cluster_caps(int caps[4]);
// out[M][n_out] = silu(x.wa) * (x.wa') (SwiGLU: wa = W_gate, wb = W_up) or
// x.wa (+ resid) (plain: wa = W_down, wb unused).  `counters`: n_cb arrival
// counters, zero on entry when `counters_clean` (left so by the previous call
// on the same stream), else cleared first.
// The FP8 up projection: x and the weights are e4m3 codes (the weights
// [n_out, K], kWeightsNK), and each f32 sum (row i, column j) is multiplied by
// sx[i] * sw_a[j] (gate) or sx[i] * sw_b[j] (up).  The tensor maps view each
// 8-bit matrix as a 16-bit one of half the columns, so K is passed as the
// number of byte pairs (a 128-byte k-block holds 128 e4m3 values).
struct Fp8Scales {
  const float* sx;     // [M]
  const float* sw_a;   // [n_out], gate
  const float* sw_b;   // [n_out], up
};

// wlayout: a WeightLayout.  fp8: null, or the FP8 scales (SwiGLU mode only).
cudaError_t launch_skinny_tc(const void* x, const void* wa, const void* wb, void* out,
                             const void* resid, int64_t M, int64_t K, int64_t n_out,
                             int wlayout, const SkinnyPlan& p, float* part,
                             unsigned* counters, bool counters_clean, unsigned* status,
                             uint64_t timeout_ns, cudaStream_t st,
                             const Fp8Scales* fp8 = nullptr);
constexpr size_t kStreamCounterBytes = 64 * 1024;   // per-stream arrival counters

// Tile tensor-core path (bf16, large M): 128-row output tiles.  SwiGLU:
// 128 output columns whose gate and up accumulators sit side by side
// (128 x 256 f32), SwiGLU applied before the bf16 store.  Plain (down
// projection): 256 output columns, + residual, bf16 store.
// With `pair`, a tile is 256 rows computed by a 2-CTA cluster (cta_group::2
// MMAs); n_mb then counts 256-row blocks and grid is even.  Tiles from
// dp_tiles on form a stream-K tail (sk_iters > 0): their (tile, k-block)
// iterations are shared out evenly over the grid's units, and partial tiles
// meet in `part_bytes` of f32 slots with `counters_bytes` of arrival counters.
// With `seq` (single-CTA SwiGLU tiles only), a tile runs a k loop over W_gate
// and then one over W_up, each of N = 128.
struct TilePlan {
  int64_t n_mb, n_nb, n_kb, tiles;
  int grid;
  bool plain;
  bool pair;
  bool seq;    // SwiGLU: gate then up k loops (N = 128 each) instead of one N = 256 loop
  int64_t band;   // row blocks per band of the tile order (n_mb: one band)
  int64_t dp_tiles, sk_iters, sk_q, sk_r;
  size_t counters_bytes, part_bytes;
};
// max_pairs: 2-CTA clusters of the tile kernel that fit on the device at once.
TilePlan plan_tile(int64_t M, int64_t K, int64_t n_out, int num_sms, bool plain,
                   int max_pairs, const Tuning& tn = Tuning{});
cudaError_t tile_max_pairs(int* pairs);
cudaError_t launch_tile_tc(const void* x, const void* wa, const void* wb, void* out,
                           const void* resid, int64_t M, int64_t K, int64_t n_out,
                           int wlayout, const TilePlan& p, float* part, unsigned* counters,
                           bool counters_clean, unsigned* status, uint64_t timeout_ns,
                           cudaStream_t st, const Fp8Scales* fp8 = nullptr);

// FP8 quantization (e4m3; multiplier 448 / amax, scale amax / 448):
// x [M, K] bf16 -> codes [M, K] and per-row scales; w [K, N] bf16 -> codes
// [N, K] (transposed) and per-column scales (amax_scratch: N unsigned).
cudaError_t launch_quantize_rows_fp8(const void* x, void* codes, float* scales, int64_t M,
                                     int64_t K, cudaStream_t st);
cudaError_t launch_quantize_cols_fp8(const void* w, void* codes_nk, float* scales,
                                     unsigned* amax_scratch, int64_t K, int64_t N,
                                     int num_sms, cudaStream_t st);

}  // namespace swg
