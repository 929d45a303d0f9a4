// Skinny-M path on the tensor cores (bf16, M <= 256): one kernel, split-K,
// deterministic in-kernel reduction, SwiGLU applied after the sums complete.
//
// The decode-time product of "Ou part le temps d'un token" ("Un kernel pour
// les matrices etroites") has too few output rows to fill the GPU, so the
// work is cut along the weights: the grid is split over (64-column block,
// 64-deep k block) units of W_gate/W_up, and the shared dimension K is split
// among CTAs so that every SM streams the same amount of weight bytes.
// Partial sums of each column block are combined in a fixed order (by k),
// never with atomics into the output, so a call's result is reproducible bit
// for bit, as that section requires.  As in its slice-reduction pass
// ("Deux operations de trop" puts the bias there), the element-wise work --
// here silu(g) * u -- runs only once the sums are complete.
//
// GB300 design (not the page's SIMT kernel):
//   * swap-AB tcgen05 MMA: A = a 128-row tile made of 64 W_gate columns and
//     the same 64 W_up columns (the gate/up column interleave of the SwiGLU
//     paper's Kernel-2, done per 64-column tile while loading, so W_gate and
//     W_up stay separate row-major arrays), MN-major from shared memory;
//     B = x^T, K-major, N = M rounded up (rows past M are zero-filled by TMA);
//     the accumulator D^T [128 x N] f32 lives in TMEM;
//   * TMA loads into an 8-12 stage shared-memory ring keep ~150-200 KB of
//     weight reads in flight per SM (Little's law at ~45 GB/s per SM);
//   * a persistent grid of one CTA per SM gets an equal share of units
//     (stream-K-style partition), so no SM idles at the tail;
//   * each CTA writes one f32 partial per column block it touched; the CTA
//     that finishes a column block last (an arrival counter, no waiting) sums
//     the partials in contributor order -- i.e. in k order -- applies
//     silu(g) * u and stores h as bf16.
//
// Cluster mode, for small weights (at most 32 MB, e.g. d = 896, d_ff = 4864):
// each column group is one thread-block cluster of S CTAs that split K
// evenly, S the largest size whose clusters all run at once.  Every CTA stages its finished
// accumulator in its own shared memory; after a cluster barrier the CTAs
// split the outputs, and each reads the S partial sums of its share through
// distributed shared memory, adds them in rank order (= k order, so the
// result is reproducible), applies the epilogue and stores.  No global workspace, no counters, no memset: the
// reduction never leaves the chip, which shortens the per-call critical path
// that dominates such small calls.
//
// Variants of the same kernel: the plain epilogue (down projection, plus the
// residual); [n_out, K] weights (the A operand K-major); a packed gate/up
// matrix (other box columns); and e4m3 operands (FP8: kind::f8f6f4 MMAs and
// scaled sums, a template parameter).
//
// The same kernel serves the down projection y = h . W_down (+ residual)
// ("1 . Anatomie d'un transformeur sur GPU", section 1.6, kernels #10 and
// #11) in its plain epilogue mode: an MMA tile then holds 128 adjacent W_down
// columns, and the final reduction adds the residual instead of applying
// SiLU * up.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues
// MMAs (warp 1 owns the TMEM allocation), warps 2-5 drain the accumulator.
// Every mbarrier wait is bounded; on timeout the CTA raises the device error
// word, stops, lets its in-flight copies and MMAs finish, frees TMEM and exits.
#include <atomic>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {
namespace {

using namespace tc;

constexpr int kBK = 64;                               // k per stage (128-byte rows)
constexpr int kCB = 64;                               // columns of one weight box
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
// Warp whose lane 0 issues the L2 prefetch before the dependency wait: the
// first epilogue warp, idle until the first accumulator is full.  Issued by
// the TMA producer instead, the prefetch held it back from the wait for up
// to 5 us when the TMA unit was busy (per-CTA %globaltimer trace), and the
// main loop started late.  Measured, calls back to back, 2 GiB of weights
// rotating: d = 4096 up projection, packed, M = 1 / 2 / 4: 36.9 / 37.1 /
// 36.9 us against 38.4 / 38.4 / 38.1.
constexpr int kPrefetchWarp = 2;
constexpr uint32_t kChunkBytes = kCB * kBK * 2;       // one 64 x 64 bf16 weight box
constexpr uint32_t kSubBytes = 2 * kChunkBytes;       // gate box + up box = one MMA A tile
constexpr uint32_t kPrefetchBytes = 512u * 1024u;     // weight bytes per CTA prefetched before the wait
constexpr uint32_t kRingBudget = 200u * 1024u;        // shared memory for the stage ring
// The decode rows' configuration (N = 16, two 64-column blocks per unit)
// streams best with 4 stages of 34 KB in flight per SM rather than 5 or 6
// (measured, 2 GiB of weights rotating, d = 4096: the up projection at
// M = 1 / 16 takes 38.5 / 39.0 us with 4 stages, 39.0 / 39.4 with 5, 41.0 /
// 41.2 with 6; the down projection M = 1 / 16: 22.3 / 22.5 against 22.7 /
// 22.9); at N = 32 five stages lead (40.9 against 41.4 us with 3).
constexpr uint32_t kRingBudgetN16 = 140u * 1024u;
// Rows for which the FP8 down projection takes 4-CTA clusters (see plan_skinny)
constexpr int64_t kPlainCluster4MinMFp8 = 16, kPlainCluster4MaxMFp8 = 64;

constexpr uint32_t pow2_at_least(uint32_t v, uint32_t lo) {
  uint32_t r = lo;
  while (r < v) r *= 2;
  return r;
}

// N: MMA N (M of the call rounded up); NB: adjacent 64-column blocks per unit,
// so every weight row is read in NB x 128-byte contiguous runs per matrix.
// KB: 64-deep k blocks per unit (and stage); with [n_out, K] weights a unit
// then reads KB x 128 contiguous bytes of every weight row it covers.
template <int N, int NB, int KB = 1>
struct SkCfg {
  static constexpr uint32_t kBTileBytes = (uint32_t)N * kBK * 2;
  static constexpr uint32_t kKBlockBytes = NB * kSubBytes + kBTileBytes;   // one k block
  static constexpr uint32_t kStageBytes = KB * kKBlockBytes;
  static constexpr int kFit =
      (int)(((N == 16 && NB == 2 && KB == 1) ? kRingBudgetN16 : kRingBudget) / kStageBytes);
  static constexpr int kStages = kFit > 12 ? 12 : kFit;
  static constexpr uint32_t kAccCols = (uint32_t)NB * N;          // one accumulator buffer
  static constexpr uint32_t kTmemCols = pow2_at_least(2 * kAccCols, 32);
  static constexpr uint32_t kRingBytes = (uint32_t)kStages * kStageBytes;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kRingBytes + 512;
  static_assert(2 * kAccCols <= 512, "accumulators exceed TMEM");
  // cluster mode stages one accumulator (NB x N x 128 f32) in the idle ring
  static_assert((size_t)NB * N * 128 * 4 <= (size_t)kStages * kStageBytes, "ring too small");
  static_assert(kStages >= 2, "stage too large");
};

struct SkArgs {
  int M, n_out, n_kb, maxq;   // n_out: output columns (d_ff, or d for the down projection)
  int64_t units;
  int grid;
  int hint;             // 1: weight loads carry an L2 evict_first hint
  int kmajor;           // weights stored [n_out, K] (K contiguous) instead of [K, n_out]
  int packed;           // SwiGLU: one packed gate/up matrix (tm_wg = tm_wu)
  const float* sx;      // fp8: [M] row scales of x
  const float* sw_a;    // fp8: [n_out] column scales of W_gate
  const float* sw_b;    // fp8: [n_out] column scales of W_up
  int prefetch_units;   // units each CTA prefetches into L2 before the dependency wait
  int cluster;          // cluster mode: CTAs per column group (0: stream-K mode)
  int bulk;             // stream-K: final sums staged by bulk copies when the ring is idle
  int split;            // stream-K: write the partial sums only (skinny_sum_kernel adds them)
  int nb;               // 64-column blocks per unit (the sum kernel's slot layout)
  int release_early;    // the sum kernel releases the next kernel before its wait
  int k64;              // 64-deep k blocks of K (a unit's k blocks past it are skipped)
  float* part;          // [n_cg][maxq][NB][2][M][64]
  unsigned* counters;   // [n_cg], zero on entry, zero again on exit
  uint16_t* out;        // [M][n_out] bf16
  const uint16_t* resid;   // plain mode: [M][n_out] bf16 added to the sums, or null
  unsigned* status;
  uint64_t timeout_ns;
};

// Epilogue modes.  kSwiGLU: A tile = 64 W_gate columns over the same 64 W_up
// columns, output = silu(g) * u for 64 columns.  kPlain: A tile = 128
// adjacent columns of one weight, output = sum (+ residual) for 128 columns.
constexpr int kSwiGLU = 0;
constexpr int kPlain = 1;

// CTA whose unit range [c U / G, (c+1) U / G) contains unit t.
__device__ __forceinline__ int64_t cta_of(int64_t t, int64_t U, int64_t G) {
  return ((t + 1) * G + U - 1) / U - 1;
}

// FP8, plain mode: the sums of row m, columns col..col+3 times sx[m] sw[col..].
__device__ __forceinline__ void fp8_scale1(float4& g, const SkArgs& a, int m, int64_t col) {
  const float sxm = a.sx[m];
  const float4 sw = *reinterpret_cast<const float4*>(a.sw_a + col);
  g.x *= sxm * sw.x; g.y *= sxm * sw.y; g.z *= sxm * sw.z; g.w *= sxm * sw.w;
}

// FP8: the sums of row m, columns col..col+3 times sx[m] sw[col..].
__device__ __forceinline__ void fp8_scale(float4& g, float4& u, const SkArgs& a, int m,
                                          int64_t col) {
  const float sxm = a.sx[m];
  const float4 sg = *reinterpret_cast<const float4*>(a.sw_a + col);
  const float4 su = *reinterpret_cast<const float4*>(a.sw_b + col);
  g.x *= sxm * sg.x; g.y *= sxm * sg.y; g.z *= sxm * sg.z; g.w *= sxm * sg.w;
  u.x *= sxm * su.x; u.y *= sxm * su.y; u.z *= sxm * su.z; u.w *= sxm * su.w;
}

// Output columns col..col+3 of row m from their finished sums g (and u):
// FP8 sums scaled first; then silu(g) * u (SwiGLU) or g + residual (plain);
// stored as bf16.
// `rsrc`: where the residual's 4 values are (a copy in shared memory), or
// null to read them from a.resid.
template <int MODE, bool FP8>
__device__ __forceinline__ void store_chunk(const SkArgs& a, float4 g, float4 u, int m,
                                            int64_t col, const uint16_t* rsrc = nullptr) {
  const int64_t o = (int64_t)m * a.n_out + col;
  uint2 ov;
  if constexpr (MODE == kSwiGLU) {
    if constexpr (FP8) fp8_scale(g, u, a, m, col);
    ov.x = pack_bf16x2(silu_fast(g.x) * u.x, silu_fast(g.y) * u.y);
    ov.y = pack_bf16x2(silu_fast(g.z) * u.z, silu_fast(g.w) * u.w);
  } else {
    if constexpr (FP8) fp8_scale1(g, a, m, col);
    if (a.resid) {
      const uint2 rv = *reinterpret_cast<const uint2*>(rsrc ? rsrc : a.resid + o);
      g.x += bf16_lo(rv.x); g.y += bf16_hi(rv.x);
      g.z += bf16_lo(rv.y); g.w += bf16_hi(rv.y);
    }
    ov.x = pack_bf16x2(g.x, g.y);
    ov.y = pack_bf16x2(g.z, g.w);
  }
  *reinterpret_cast<uint2*>(a.out + o) = ov;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, unsigned* status,
                                           uint64_t timeout_ns) {
  int never = 0;
  return mbar_wait(bar, parity, &never, status, timeout_ns);
}

// FP8: e4m3 operands (kind::f8f6f4) and scaled sums.  A compile-time choice:
// one kernel issuing MMAs of two kinds behind a runtime branch measured
// 20-40 % slower on its bf16 work.
template <int N, int NB, int MODE, bool FP8, int KB>
__global__ void __launch_bounds__(kThreads, 1)
skinny_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_wg,
                 const __grid_constant__ CUtensorMap tm_wu, const SkArgs a) {
  using C = SkCfg<N, NB, KB>;
  // Weight columns of one unit's sub-block, and where its two 64-column
  // boxes come from: (tm_wg, col) and (tm_wu, col) for SwiGLU, (tm_wg, col)
  // and (tm_wg, col + 64) for the plain mode.
  // A packed gate/up matrix holds gate block b at column 2 col and up block
  // b at 2 col + 64, both in tm_wg (the plain mode's pattern at twice the
  // column).
  constexpr int kSubCols = MODE == kSwiGLU ? kCB : 2 * kCB;
  const CUtensorMap* hi_map = (MODE == kSwiGLU && !a.packed) ? &tm_wu : &tm_wg;
  const int kHiOff = (MODE == kSwiGLU && !a.packed) ? 0 : kCB;
  const int col_mul = (MODE == kSwiGLU && a.packed) ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* rbar = drain + 1;   // [2]: bulk-copied partial sums landed (final sums)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ticket = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = a.units, G = a.grid, c = blockIdx.x;
  // Stream-K mode: an even share of the (group, k-block) units.  Cluster mode:
  // CTA rank r of cluster g takes k-blocks [r n_kb / S, (r+1) n_kb / S) of
  // column group g (S <= n_kb, so every CTA has at least one).
  int64_t u0 = c * U / G, u1 = (c + 1) * U / G;
  const int S = a.cluster;
  const int64_t cgroup = S ? c / S : 0;
  const int crank = S ? (int)(c % S) : 0;
  if (S) {
    u0 = cgroup * a.n_kb + (int64_t)crank * a.n_kb / S;
    u1 = cgroup * a.n_kb + (int64_t)(crank + 1) * a.n_kb / S;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], kEpiThreads);
    mbar_init(&tempty[1], kEpiThreads);
    mbar_init(drain, 1);
    mbar_init(&rbar[0], 1);
    mbar_init(&rbar[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything above overlaps the previous kernel's tail.  So does an L2
  // prefetch of this CTA's first weight boxes and of the x boxes they meet: a
  // prefetch only reads, and L2 is where every later write lands, so it is
  // safe before the wait.  From
  // the wait on, the kernel reads x and the workspace, which the previous
  // kernel may still be writing.
  if (warp == kPrefetchWarp && lane == 0) {
    const int64_t pend = min(u1, u0 + (int64_t)a.prefetch_units);
    for (int64_t t = u0; t < pend; ++t) {
      const int cg = (int)(t / a.n_kb), kbu = (int)(t - (int64_t)cg * a.n_kb);
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        const int kb = kbu * KB + j;
        if (KB > 1 && kb >= a.k64) break;
        // x too: the same argument holds, and a call whose x was evicted
        // since it was written would otherwise wait a DRAM round trip for
        // its first stage (the d = 4096 decode sweep, M = 1 ... 16 in turn:
        // 0.4-0.6 % per step)
        tma_prefetch_l2_2d(&tm_x, kb * kBK, 0);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const int col = (cg * NB + b) * kSubCols * col_mul;
          if (a.kmajor) {
            tma_prefetch_l2_2d(&tm_wg, kb * kBK, col);
            tma_prefetch_l2_2d(hi_map, kb * kBK, col + kHiOff);
          } else {
            tma_prefetch_l2_2d(&tm_wg, col, kb * kBK);
            tma_prefetch_l2_2d(hi_map, col + kHiOff, kb * kBK);
          }
        }
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t evict_first = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = u0; t < u1; ++t) {
        const int cg = (int)(t / a.n_kb), kbu = (int)(t - (int64_t)cg * a.n_kb);
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
          ok = false;
          break;
        }
        uint8_t* st = stages + (size_t)stage * C::kStageBytes;
        // k blocks of this unit inside K (a unit of KB > 1 blocks may end past it)
        const int nkb = KB > 1 ? min(KB, a.k64 - kbu * KB) : 1;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)nkb * C::kKBlockBytes);
#pragma unroll
        for (int j = 0; j < KB; ++j) {
          if (j >= nkb) break;
          const int kb = kbu * KB + j;
          uint8_t* sk = st + j * C::kKBlockBytes;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const int col = (cg * NB + b) * kSubCols * col_mul;
            uint8_t* sb = sk + b * kSubBytes;
            // [K, n_out] weights: box (col, k); [n_out, K] weights: box (k, col).
            const int c0 = a.kmajor ? kb * kBK : col, c1 = a.kmajor ? col : kb * kBK;
            const int h0 = a.kmajor ? kb * kBK : col + kHiOff, h1 = a.kmajor ? col + kHiOff : kb * kBK;
            if (a.hint) {
              tma_load_2d_hint(sb, &tm_wg, &full[stage], c0, c1, evict_first);
              tma_load_2d_hint(sb + kChunkBytes, hi_map, &full[stage], h0, h1, evict_first);
            } else {
              tma_load_2d(sb, &tm_wg, &full[stage], c0, c1);
              tma_load_2d(sb + kChunkBytes, hi_map, &full[stage], h0, h1);
            }
          }
          tma_load_2d(sk + NB * kSubBytes, &tm_x, &full[stage], kb * kBK, 0);
        }
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's memory goes away
        const int64_t first = issued > C::kStages ? issued - C::kStages : 0;
        for (int64_t i = first; i < issued; ++i)
          wait_drain(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), a.status,
                     a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // A (the weight tile) is MN-major for [K, n_out] weights, K-major for
      // [n_out, K] weights; B (x^T) is always K-major.
      // (FP8: e4m3 codes, K-major; one MMA takes 32 of them, the same 32 bytes)
      const uint32_t idesc = FP8        ? idesc_e4m3_f32(128, N)
                             : a.kmajor ? idesc_bf16_f32(128, N, false, false)
                                        : idesc_bf16_f32(128, N, true, false);
      // per 16-deep k step: MN-major tiles advance 16 rows of 128 bytes (two
      // swizzle atoms; the two 64-column boxes are kChunkBytes apart), K-major
      // tiles 32 bytes along their 128-byte rows (8-row groups 1024 B apart).
      const uint32_t a_step = a.kmajor ? 32u : 2048u;
      const uint32_t a_lbo = a.kmajor ? 16u : kChunkBytes;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int64_t t = u0;
      while (ok && t < u1) {
        const int64_t cg = t / a.n_kb;
        const int64_t seg_end = min(u1, (cg + 1) * (int64_t)a.n_kb);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int64_t tt = t; tt < seg_end; ++tt) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nkb = KB > 1 ? min(KB, a.k64 - (int)(tt - cg * a.n_kb) * KB) : 1;
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            if (j >= nkb) break;
            const uint32_t s_addr =
                smem_u32(stages + (size_t)stage * C::kStageBytes + j * C::kKBlockBytes);
            const uint32_t b_addr = s_addr + NB * kSubBytes;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const uint32_t d_tmem = tmem + (uint32_t)(acc * C::kAccCols + b * N);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                // A: 16 k-rows further down the MN-major tile (2 swizzle atoms);
                // B: 32 bytes further along the K-major 128-byte rows.
                const uint64_t ad =
                    smem_desc_sw128(s_addr + b * kSubBytes + kk * a_step, a_lbo, 1024u);
                const uint64_t bd = smem_desc_sw128(b_addr + kk * 32u, 16u, 1024u);
                const uint32_t accum = (tt != t || j != 0 || kk != 0) ? 1u : 0u;
                if constexpr (FP8)
                  mma_e4m3(d_tmem, ad, bd, idesc, accum);
                else
                  mma_bf16(d_tmem, ad, bd, idesc, accum);
              }
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
        t = seg_end;
      }
      // every MMA this thread issued completes before TMEM is released
      mma_commit(drain);
      wait_drain(drain, 0, a.status, a.timeout_ns);
    }
    __syncwarp();
  } else if (S) {
    // ---------------- cluster mode: stage this CTA's sums ----------------
    // The accumulator is complete once tfull fires; every MMA has then read
    // its operands, so the ring is idle and holds the sums as P[b][m][row].
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    float* xb = reinterpret_cast<float*>(stages);
    if (mbar_wait(&tfull[0], 0, abort_flag, a.status, a.timeout_ns)) {
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int ch = 0; ch < N / 16; ++ch) {
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * N + ch * 16), r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            xb[(size_t)(b * N + ch * 16 + i) * 128 + row] = __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int quarter = warp & 3;          // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;   // tile row: 0..63 gate, 64..127 up
    const int gu = row >> 6, j = row & 63;
    const int et = threadIdx.x - 64;       // 0..127
    const int64_t Mrow = (int64_t)a.M * kCB;     // floats of one [M][64] partial block
    constexpr int kGroupCols = NB * kSubCols;    // output columns of one unit group
    int acc = 0;
    uint32_t acc_phase = 0;
    int64_t t = u0;
    while (t < u1) {
      const int64_t cg = t / a.n_kb;
      const int64_t seg_end = min(u1, (cg + 1) * (int64_t)a.n_kb);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, a.status, a.timeout_ns)) break;
      tc_fence_after();
      const int64_t c_lo = cta_of(cg * a.n_kb, U, G);
      const int64_t c_hi = cta_of((cg + 1) * a.n_kb - 1, U, G);
      const int n_contrib = (int)(c_hi - c_lo + 1);
      float* slot = a.part + (cg * a.maxq + (c - c_lo)) * NB * 2 * Mrow;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int ch = 0; ch < N / 16; ++ch) {
          uint32_t r[16];
          tmem_ld_x16(tmem + ((uint32_t)(quarter * 32) << 16) +
                          (uint32_t)(acc * C::kAccCols + b * N + ch * 16), r);
          tmem_wait_ld();
          float* sb = slot + (int64_t)(b * 2 + gu) * Mrow;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = ch * 16 + i;
            if (m < a.M) sb[(int64_t)m * kCB + j] = __uint_as_float(r[i]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      // Two-kernel form: the sums are added by skinny_sum_kernel, which the
      // end of this grid releases.
      if (a.split) {
        t = seg_end;
        continue;
      }
      // The CTA that completes column group cg last reduces it.
      __syncwarp();
      named_bar_sync(1, kEpiThreads);
      if (et == 0) {
        __threadfence();
        *ticket = (int)atomicAdd(&a.counters[cg], 1u);
      }
      __syncwarp();
      named_bar_sync(1, kEpiThreads);
      const int tk = *ticket;
      if (tk == n_contrib - 1) {
        __threadfence();
        const float* pg = a.part + cg * a.maxq * NB * 2 * Mrow;
        const int64_t q_stride = (int64_t)NB * 2 * Mrow;   // floats of one slot
        constexpr int kChunks = kGroupCols / 4;      // 4-column chunks per row of the group
        // When this group is the CTA's last segment, every MMA of the CTA has
        // completed (tfull fired) and no copy is pending, so the stage ring
        // is idle: the partial sums (and the residual rows) are staged there
        // by bulk copies, issued all at once, instead of being read from L2
        // a few loads per thread per round trip.  Passes of R rows; with
        // more than one pass, two half-ring buffers alternate so that the
        // next pass lands while this one is summed.  The sums run in slot
        // (= k) order, as in the L2 path below: same bits either way.
        const bool plain_resid = MODE == kPlain && a.resid != nullptr;
        const int blocks = n_contrib * NB * 2;           // [M][64] blocks of the group
        const uint32_t row_bytes = (uint32_t)blocks * kCB * 4 + (plain_resid ? kGroupCols * 2 : 0);
        int R = 0, npass = 0;
        uint32_t buf_bytes = 0;
        if (a.bulk && seg_end == u1) {
          if ((uint64_t)a.M * row_bytes <= C::kRingBytes) {
            R = a.M;
            buf_bytes = C::kRingBytes;
          } else {
            buf_bytes = (C::kRingBytes / 2) & ~127u;
            R = (int)(buf_bytes / row_bytes);
          }
          npass = R > 0 ? (a.M + R - 1) / R : 0;
        }
        if (npass > 0) {
          const int64_t cbase = cg * kGroupCols;
          const int ccols = (int)min((int64_t)kGroupCols, (int64_t)a.n_out - cbase);
          const uint32_t resid_off = (uint32_t)blocks * R * kCB * 4;
          // pass p -> buffer p & 1, issued by warp 2 (et 0..31)
          auto issue = [&](int pp) {
            const int b = pp & 1;
            uint8_t* buf = stages + (size_t)b * buf_bytes;
            const int m0 = pp * R, nr = min(R, a.M - m0);
            const int n_copies = blocks + (plain_resid ? nr : 0);
            if (lane == 0)
              mbar_arrive_expect_tx(&rbar[b], (uint32_t)blocks * nr * kCB * 4 +
                                                  (plain_resid ? (uint32_t)(nr * ccols * 2) : 0u));
            __syncwarp();
            fence_async_global();
            for (int i = lane; i < n_copies; i += 32) {
              if (i < blocks) {
                const int q = i / (NB * 2), bb = i - q * (NB * 2);
                bulk_load_g2s(buf + (size_t)i * R * kCB * 4,
                              pg + q * q_stride + bb * Mrow + (int64_t)m0 * kCB,
                              (uint32_t)nr * kCB * 4, &rbar[b]);
              } else {
                const int r = i - blocks;
                bulk_load_g2s(buf + resid_off + (size_t)r * kGroupCols * 2,
                              a.resid + (int64_t)(m0 + r) * a.n_out + cbase,
                              (uint32_t)ccols * 2, &rbar[b]);
              }
            }
          };
          if (et < 32) {
            issue(0);
            if (npass > 1) issue(1);
          }
          int issued = npass > 1 ? 2 : 1;
          int done = 0;
          bool failed = false;
          for (int pp = 0; pp < npass; ++pp) {
            const int b = pp & 1;
            // every epilogue thread reaches the barrier below, waited or not
            if (failed || !mbar_wait(&rbar[b], (uint32_t)((pp >> 1) & 1), abort_flag, a.status,
                                     a.timeout_ns))
              failed = true;
            else
              done = pp + 1;
            const uint8_t* buf = stages + (size_t)b * buf_bytes;
            const float* fb = reinterpret_cast<const float*>(buf);
            const int m0 = pp * R, nr = min(R, a.M - m0);
            for (int idx = failed ? nr * kChunks : et; idx < nr * kChunks; idx += kEpiThreads) {
              const int ml = idx / kChunks, ch = idx - ml * kChunks;
              const int blk = MODE == kSwiGLU ? (ch >> 4) * 2 : (ch >> 4);
              const float* b0 = fb + ((size_t)blk * R + ml) * kCB + (ch & 15) * 4;
              float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
              for (int q = 0; q < n_contrib; ++q) {   // slot order = k order
                const float* bq = b0 + (size_t)q * NB * 2 * R * kCB;
                const float4 v = *reinterpret_cast<const float4*>(bq);
                g.x += v.x; g.y += v.y; g.z += v.z; g.w += v.w;
                if constexpr (MODE == kSwiGLU) {
                  const float4 w = *reinterpret_cast<const float4*>(bq + (size_t)R * kCB);
                  u.x += w.x; u.y += w.y; u.z += w.z; u.w += w.w;
                }
              }
              const int64_t col = cbase + ch * 4;
              if (col < a.n_out) {
                const uint16_t* rs =
                    plain_resid ? reinterpret_cast<const uint16_t*>(buf + resid_off +
                                                                    (size_t)ml * kGroupCols * 2) +
                                      ch * 4
                                : nullptr;
                store_chunk<MODE, FP8>(a, g, u, m0 + ml, col, rs);
              }
            }
            named_bar_sync(1, kEpiThreads);   // buffer b has been read by all
            if (pp + 2 < npass) {
              // one decision for the whole issuing warp
              const int stop = et < 32 ? __shfl_sync(0xffffffffu, (int)*abort_flag, 0) : 1;
              if (et < 32 && !stop) {
                issue(pp + 2);
                ++issued;
              }
            }
          }
          // after a timeout: let the copies still in flight land before the
          // CTA's shared memory goes away
          for (int pp = done; pp < issued; ++pp)
            wait_drain(&rbar[pp & 1], (uint32_t)((pp >> 1) & 1), a.status, a.timeout_ns);
          if (et == 0) a.counters[cg] = 0u;   // ready for the next call
          t = seg_end;
          continue;
        }
        // Each thread sums 4 adjacent output columns of one row at a time:
        // 16-byte loads, several outputs in flight together.  SwiGLU: gate
        // and up partials of the same columns; plain: one partial per column.
        const int total = a.M * kChunks;
        // The sums are bound by L2 latency, not bandwidth: each round of loads
        // waits one L2 round trip.  So a round loads kQ slots' partials of
        // kBatch chunks (twice that for SwiGLU) before it adds any of them.
        constexpr int kBatch = 4;
        constexpr int kQ = MODE == kSwiGLU ? 2 : 4;
        for (int base = et; base < total; base += kBatch * kEpiThreads) {
          float4 g[kBatch], u[kBatch];
          int off[kBatch];
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            g[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            u[i] = g[i];
            const int idx = base + i * kEpiThreads;
            const int id = idx < total ? idx : 0;    // a chunk past the end reads chunk 0, unused
            const int m = id / kChunks, ch = id - m * kChunks;
            // SwiGLU: chunk ch -> sub-block ch/16, gate half; plain: sub-block
            // ch/32, half (ch/16)&1.  Either way (ch >> 4) picks the [M][64]
            // partial block in [NB][2] order.
            const int blk = MODE == kSwiGLU ? (ch >> 4) * 2 : (ch >> 4);
            off[i] = blk * (int)Mrow + m * kCB + (ch & 15) * 4;
          }
          // slot q holds CTA (c_lo + q)'s sums; adding in q order is k order
          for (int q0 = 0; q0 < n_contrib; q0 += kQ) {
            float4 vg[kQ][kBatch], vu[kQ][kBatch];
#pragma unroll
            for (int j = 0; j < kQ; ++j) {
              const bool have = q0 + j < n_contrib;
              const float* pq = pg + (int64_t)(q0 + j) * q_stride;
#pragma unroll
              for (int i = 0; i < kBatch; ++i) {
                vg[j][i] = have ? __ldcg(reinterpret_cast<const float4*>(pq + off[i]))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (MODE == kSwiGLU)
                  vu[j][i] = have ? __ldcg(reinterpret_cast<const float4*>(pq + off[i] + Mrow))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
#pragma unroll
            for (int j = 0; j < kQ; ++j) {
              if (q0 + j < n_contrib) {
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                  g[i].x += vg[j][i].x; g[i].y += vg[j][i].y;
                  g[i].z += vg[j][i].z; g[i].w += vg[j][i].w;
                  if constexpr (MODE == kSwiGLU) {
                    u[i].x += vu[j][i].x; u[i].y += vu[j][i].y;
                    u[i].z += vu[j][i].z; u[i].w += vu[j][i].w;
                  }
                }
              }
            }
          }
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            const int idx = base + i * kEpiThreads;
            if (idx >= total) continue;
            const int m = idx / kChunks, ch = idx - m * kChunks;
            const int64_t col = cg * kGroupCols + ch * 4;
            // n_out is a multiple of 8: a chunk is all in or all out
            if (col < a.n_out) store_chunk<MODE, FP8>(a, g[i], u[i], m, col);
          }
        }
        if (et == 0) a.counters[cg] = 0u;   // ready for the next call
      } else if (tk >= n_contrib) {
        // the counter did not start at zero: report it and leave it clean
        if (et == 0) {
          atomicOr(a.status, kStatusStaleCounter);
          a.counters[cg] = 0u;
        }
      }
      t = seg_end;
    }
    __syncwarp();
  }

  if (S) {
    // ---------------- cluster mode: the cluster reduces ----------------
    // The CTAs split the group's outputs (contiguous chunk ranges) and each
    // sums its share over the S staged accumulators, so they read distributed
    // shared memory side by side instead of one CTA reading it all (d = 896
    // down projection, M = 16 / 64 / 96: 12.8 / 26.4 / 35.2 us with rank 0
    // alone, 9.4 / 11.8 / 13.5 us shared).
    cluster_sync_all();   // every CTA's sums are staged
    if (warp >= 2 && !*abort_flag) {
      constexpr int kSubCols2 = MODE == kSwiGLU ? kCB : 2 * kCB;
      constexpr int kGroupCols = NB * kSubCols2;
      constexpr int kChunks = kGroupCols / 4;
      constexpr int kMaxS = 8;
      const int et = threadIdx.x - 64;
      uint32_t base[kMaxS];
      const uint32_t local = smem_u32(stages);
#pragma unroll
      for (int r = 0; r < kMaxS; ++r) base[r] = r < S ? mapa_shared(local, (uint32_t)r) : 0u;
      const int total = a.M * kChunks;
      // R CTAs share the chunks: no more than one pass of 128 threads' worth
      // each (a call whose chunks fit one pass stays on rank 0: d = 896, up
      // projection, M = 1 measured 7.4 us that way, 7.7 us split in two).
      const int R = min(S, (total + kEpiThreads - 1) / kEpiThreads);
      const int lo = crank < R ? (int)((int64_t)crank * total / R) : 0;
      const int hi = crank < R ? (int)((int64_t)(crank + 1) * total / R) : 0;
      for (int idx = lo + et; idx < hi; idx += kEpiThreads) {
        const int m = idx / kChunks, ch = idx - m * kChunks;
        // SwiGLU: 16 chunks per 64-column sub-block, gate rows ch*4.., up rows
        // 64 + ch*4..; plain: 32 chunks per 128-column sub-block, rows ch*4..
        const int b = MODE == kSwiGLU ? (ch >> 4) : (ch >> 5);
        const int r0 = MODE == kSwiGLU ? (ch & 15) * 4 : (ch & 31) * 4;
        const uint32_t off = (uint32_t)(((b * N + m) * 128 + r0) * 4);
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
#pragma unroll
        for (int r = 0; r < kMaxS; ++r) {   // rank order = k order
          if (r < S) {
            const float4 pv = ld_shared_cluster_v4(base[r] + off);
            g.x += pv.x; g.y += pv.y; g.z += pv.z; g.w += pv.w;
            if constexpr (MODE == kSwiGLU) {
              const float4 qv = ld_shared_cluster_v4(base[r] + off + 64 * 4);
              u.x += qv.x; u.y += qv.y; u.z += qv.z; u.w += qv.w;
            }
          }
        }
        const int64_t col = cgroup * kGroupCols + ch * 4;
        if (col < a.n_out) store_chunk<MODE, FP8>(a, g, u, m, col);   // n_out: a multiple of 8
      }
    }
    __syncwarp();
    cluster_sync_all();   // each CTA keeps its shared memory until all peers are done
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Second kernel of the two-kernel form (stream-K mode): one thread per
// output chunk (4 adjacent columns of one row) adds the chunk's partial sums
// from every CTA of its column group in slot (= k) order -- the order of the
// one-kernel form's last CTA, so the bits are the same -- and applies the
// epilogue.  A thread issues all of its loads before the first add, so the
// sums take one or two L2 round trips on a grid as wide as the output,
// instead of one CTA per column group walking its slots while the rest of
// the GPU idles.  This is the slice-reduction pass of "Ou part le temps d'un
// token" (section "Un kernel pour les matrices etroites") on this kernel's
// partial-sum layout.
constexpr int kSumThreads = 256;

template <int MODE, bool FP8>
__global__ void __launch_bounds__(kSumThreads) skinny_sum_kernel(const SkArgs a) {
  // Launched with programmatic serialisation behind the GEMM: its partial
  // sums are complete and visible once that grid is (the dependency wait).
  // With release_early the next kernel in the stream may launch at once (its
  // own dependency wait still covers this grid's completion): an FP8 call
  // starts with its activation quantizer, and releasing it early lets the
  // next call's GEMM take the SMs this call's GEMM frees, and prefetch its
  // weights, one launch sooner.  Measured, FP8 down projection d = 4096,
  // M = 4 / 8: 16.9 / 17.0 us against 18.7 / 18.8 without (one-kernel form
  // 17.4 / 18.0).  The bf16 down projection with 256-column groups gains
  // too once the next GEMM prefetches more (see plan_skinny).
  if (a.release_early) pdl_launch_dependents();
  // Everything up to the wait reads only the kernel's parameters: the
  // chunk's index arithmetic (64-bit divisions, long enough to matter here:
  // a per-CTA %globaltimer trace put this kernel at 1.8-3.4 us from its wait
  // to its stores at M = 1) and an L2 prefetch of the residual and the
  // column scales, which are inputs of the call like the weights.
  constexpr int kSubCols = MODE == kSwiGLU ? kCB : 2 * kCB;
  constexpr int kBatch = MODE == kSwiGLU ? 6 : 12;   // slots loaded per round
  const int64_t group_cols = (int64_t)a.nb * kSubCols;
  const int64_t cpr = a.n_out / 4;                    // chunks per row (n_out % 8 == 0)
  const int64_t idx = (int64_t)blockIdx.x * kSumThreads + threadIdx.x;
  if (idx >= (int64_t)a.M * cpr) return;
  const int m = (int)(idx / cpr);
  const int64_t col = (idx - (int64_t)m * cpr) * 4;
  const int64_t cg = col / group_cols;
  const int ch = (int)((col - cg * group_cols) / 4);
  const int64_t U = a.units, G = a.grid;
  const int64_t c_lo = cta_of(cg * a.n_kb, U, G);
  const int n_contrib = (int)(cta_of((cg + 1) * a.n_kb - 1, U, G) - c_lo + 1);
  const int64_t Mrow = (int64_t)a.M * kCB;            // floats of one [M][64] block
  const int64_t q_stride = (int64_t)a.nb * 2 * Mrow;  // floats of one slot
  // the chunk's [M][64] block in [NB][2] order: SwiGLU -> sub-block ch/16,
  // gate half (up at + Mrow); plain -> sub-block ch/32, half (ch/16) & 1
  const int blk = MODE == kSwiGLU ? (ch >> 4) * 2 : (ch >> 4);
  const float* p0 = a.part + cg * a.maxq * q_stride + blk * Mrow + (int64_t)m * kCB + (ch & 15) * 4;
  const int64_t o = (int64_t)m * a.n_out + col;
  if (MODE == kPlain && (threadIdx.x & 7) == 0) {   // 8 chunks: 64 B of residual, 128 B of scales
    if (a.resid) prefetch_l2(a.resid + o);
    if (FP8) prefetch_l2(a.sw_a + col);
  }
  pdl_wait();
  pdl_launch_dependents();
  // The residual and (FP8) the scales load with the partial sums, not after
  // them.  Measured with the changes above, FP8 down projection d = 4096,
  // calls back to back, M = 1 / 8: 15.9 / 16.5 us against 17.3 / 17.6.
  uint2 rv = make_uint2(0u, 0u);
  if (MODE == kPlain && a.resid) rv = __ldg(reinterpret_cast<const uint2*>(a.resid + o));
  float sxm = 1.f;
  float4 swv = make_float4(1.f, 1.f, 1.f, 1.f);
  if (FP8 && MODE == kPlain) {
    sxm = __ldcg(a.sx + m);
    swv = __ldcg(reinterpret_cast<const float4*>(a.sw_a + col));
  }
  float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
  for (int q0 = 0; q0 < n_contrib; q0 += kBatch) {
    float4 vg[kBatch], vu[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool have = q0 + j < n_contrib;
      const float* pq = p0 + (int64_t)(q0 + j) * q_stride;
      vg[j] = have ? __ldcg(reinterpret_cast<const float4*>(pq)) : make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (MODE == kSwiGLU)
        vu[j] = have ? __ldcg(reinterpret_cast<const float4*>(pq + Mrow))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (q0 + j < n_contrib) {
        g.x += vg[j].x; g.y += vg[j].y; g.z += vg[j].z; g.w += vg[j].w;
        if constexpr (MODE == kSwiGLU) {
          u.x += vu[j].x; u.y += vu[j].y; u.z += vu[j].z; u.w += vu[j].w;
        }
      }
    }
  }
  if constexpr (MODE == kSwiGLU) {
    store_chunk<MODE, FP8>(a, g, u, m, col);
  } else {
    // store_chunk's plain epilogue (fp8_scale1's arithmetic), with the
    // residual and the scales loaded up front
    if constexpr (FP8) {
      g.x *= sxm * swv.x; g.y *= sxm * swv.y; g.z *= sxm * swv.z; g.w *= sxm * swv.w;
    }
    if (a.resid) {
      g.x += bf16_lo(rv.x); g.y += bf16_hi(rv.x);
      g.z += bf16_lo(rv.y); g.w += bf16_hi(rv.y);
    }
    uint2 ov;
    ov.x = pack_bf16x2(g.x, g.y);
    ov.y = pack_bf16x2(g.z, g.w);
    *reinterpret_cast<uint2*>(a.out + o) = ov;
  }
}

template <int MODE, bool FP8>
cudaError_t launch_sum(const SkArgs& a, cudaStream_t st) {
  const int64_t chunks = (int64_t)a.M * (a.n_out / 4);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((chunks + kSumThreads - 1) / kSumThreads));
  cfg.blockDim = dim3(kSumThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, skinny_sum_kernel<MODE, FP8>, a);
}

template <int N, int NB, int MODE, bool FP8, int KB = 1>
cudaError_t launch_n(const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mu,
                     const SkArgs& a, cudaStream_t st) {
  using C = SkCfg<N, NB, KB>;
  auto kern = skinny_tc_kernel<N, NB, MODE, FP8, KB>;
  static std::atomic<int> configured[64];   // zero: not yet set on that device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(1, std::memory_order_release);
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.cluster ? (unsigned)a.cluster : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, mx, mg, mu, a);
}

template <int N, int MODE, bool FP8>
cudaError_t launch_nb(int nb, int kb, const CUtensorMap& mx, const CUtensorMap& mg,
                      const CUtensorMap& mu, const SkArgs& a, cudaStream_t st) {
  // two k blocks per unit: FP8 ([n_out, K] codes), one column block, N <= 64
  if constexpr (FP8 && N <= 64) {
    if (kb == 2) return nb == 1 ? launch_n<N, 1, MODE, FP8, 2>(mx, mg, mu, a, st)
                                : cudaErrorInvalidValue;
  }
  if (kb != 1) return cudaErrorInvalidValue;
  if constexpr (N <= 64) {
    if (nb == 4) return launch_n<N, 4, MODE, FP8>(mx, mg, mu, a, st);
  }
  if constexpr (N <= 128) {
    if (nb == 2) return launch_n<N, 2, MODE, FP8>(mx, mg, mu, a, st);
  }
  if (nb == 1) return launch_n<N, 1, MODE, FP8>(mx, mg, mu, a, st);
  return cudaErrorInvalidValue;
}

template <int MODE, bool FP8>
cudaError_t launch_mode(int n_pad, int nb, int kb, const CUtensorMap& mx, const CUtensorMap& mg,
                        const CUtensorMap& mu, const SkArgs& a, cudaStream_t st) {
  switch (n_pad) {
    case 16: return launch_nb<16, MODE, FP8>(nb, kb, mx, mg, mu, a, st);
    case 32: return launch_nb<32, MODE, FP8>(nb, kb, mx, mg, mu, a, st);
    case 64: return launch_nb<64, MODE, FP8>(nb, kb, mx, mg, mu, a, st);
    case 128: return launch_nb<128, MODE, FP8>(nb, kb, mx, mg, mu, a, st);
    case 256: return launch_nb<256, MODE, FP8>(nb, kb, mx, mg, mu, a, st);
    default: return cudaErrorInvalidValue;
  }
}


}  // namespace

bool skinny_plain_cluster4_fits(int64_t K, int64_t n_out, int num_sms, const int* cluster_caps) {
  const int64_t groups = (n_out + 2 * kCB - 1) / (2 * kCB);   // 128-column groups
  const int64_t cap4 = cluster_caps ? cluster_caps[2] : (int64_t)(num_sms / 4 * 0.95);
  return groups >= 1 && groups <= cap4 && (K + kBK - 1) / kBK >= 4;
}

SkinnyPlan plan_skinny(int64_t M, int64_t K, int64_t n_out, int num_sms, bool plain,
                       bool fp8, const int* cluster_caps, const Tuning& tn) {
  SkinnyPlan p{};
  int n = 16;
  while (n < M) n *= 2;
  p.n_pad = n;
  p.plain = plain;
  int nb = tn.sk_nb >= 0 ? tn.sk_nb : 2;
  if (nb != 1 && nb != 2 && nb != 4) nb = 2;
  const int64_t weight_bytes = (plain ? 1 : 2) * K * n_out * 2;
  if (plain && tn.sk_nb < 0 && weight_bytes > kSkinnyClusterMaxWeightBytes) {
    // The down projection's K is long and its output narrow, so each column
    // group collects many partial sums (stream-K mode), and the CTA that
    // completes a group adds them all while the call's other CTAs are already
    // done.  Past
    // about 256 KB of partials per group (with 256-column groups: slots x
    // 256 columns x M rows x 4 B), 128-column groups finish first, although
    // they stream the weights in shorter runs.  Measured, residual included:
    // d = 4096: 24.5 vs 26.7 us at M = 16 (180 KB), 30.4 vs 29.0 at 32
    // (360 KB), 43.5 vs 33.9 at 64; d = 8192: 79.2 vs 81.1 at M = 32
    // (196 KB), 90.2 vs 85.5 at 64.  FP8 weights stream in half the time,
    // so there the limit is half (FP8 d = 4096, M = 16: 20.6 vs 19.3 us).
    const int64_t n_kb2 = (K + kBK - 1) / kBK, n_cb2 = (n_out + 4 * kCB - 1) / (4 * kCB);
    const int64_t units2 = n_cb2 * n_kb2;
    const int64_t grid2 = units2 < num_sms ? units2 : num_sms;
    const int64_t per2 = grid2 > 0 ? units2 / grid2 : 1;
    const int64_t slots2 = per2 > 0 ? (n_kb2 + per2 - 1) / per2 + 1 : 1;
    const int64_t limit = fp8 ? (int64_t)128 << 10 : (int64_t)256 << 10;
    // With the bf16 sums in a second kernel (the default, below) no single
    // CTA reads a group's partials, and 256-column groups, whose sum kernel
    // releases the next GEMM early, lead up to 128 rows where the sums are a
    // large share of the call (measured, 2 GiB of weights rotating, d = 4096,
    // 117 MB: M = 32 / 64 / 96 / 128 take 21.7 / 23.6 / 23.5 / 24.7 us
    // against 22.7 / 24.4 / 24.9 / 25.3 with 128-column groups), and up to 64
    // rows above 256 MB (d = 8192, 484 MB: M = 64 / 128 take 76.2 / 81.8 us
    // against 77.5 / 80.1).
    const bool two_kernels = !fp8 && tn.sk_split != 0;
    const int64_t max_m2 = weight_bytes > ((int64_t)256 << 20) ? 64 : 128;
    if (two_kernels ? M > max_m2 : slots2 * 4 * kCB * 4 * M > limit) nb = 1;
  }
  // FP8 down projections of 16-64 rows: 4-CTA clusters of 128-column groups,
  // when all the groups' clusters fit at once (n_out up to 36 x 128 on
  // GB300).  The group's four K quarters then meet in distributed shared
  // memory; 128 CTAs stream the weights.  Elsewhere, and for bf16 at every
  // M, stream-K on every SM with its sums in a second kernel leads.
  // Measured, d_ff = 14336 -> d = 4096, calls back to back, 4-CTA clusters
  // against stream-K with the two-kernel sums: bf16 M = 16: 25.3 / 21.1 us;
  // 33: 26.4 / 24.1; 48: 26.8 / 26.0; 64: 27.3 / 26.1; 80: 26.7 / 26.6; 128:
  // 29.9 / 27.1; 256: 36.2 / 32.3.  FP8 M = 16: 18.0 / 18.7; 32: 18.9 /
  // 20.0; 64: 20.6 / 20.7; 96: 22.3 / 21.4; 128: 23.6 / 22.3.  (d = 8192
  // needs 64 groups, more than fit.)
  bool plain_cluster4 = false;
  if (plain && fp8 && weight_bytes > kSkinnyClusterMaxWeightBytes &&
      M >= kPlainCluster4MinMFp8 && M <= kPlainCluster4MaxMFp8 && tn.sk_nb < 0 &&
      tn.sk_cluster < 0 && skinny_plain_cluster4_fits(K, n_out, num_sms, cluster_caps)) {
    nb = 1;
    plain_cluster4 = true;
  }
  // Small weights, down projection: single 128-column groups, so twice as
  // many clusters stream the weights (measured, graph replay, d_ff = 4864 ->
  // d = 896, 8-CTA clusters: M = 1 / 16 / 64 / 128 take 7.1 / 7.5 / 8.5 /
  // 10.0 us in 7 groups against 8.3 / 8.8 / 10.9 / 14.2 us in 4).
  if (plain && weight_bytes <= kSkinnyClusterMaxWeightBytes && tn.sk_nb < 0) nb = 1;
  // Small weights, up projection, from 16 rows: single 64-column units, when
  // their twice as many column groups still fit as 2-CTA clusters at once
  // (measured, graph replay, d = 896, d_ff = 4864: M = 16 / 64 take 7.2 /
  // 8.5 us against 7.3 / 9.7 us in 128-column groups).
  if (!plain && weight_bytes <= kSkinnyClusterMaxWeightBytes && M >= 16 && tn.sk_nb < 0 &&
      tn.sk_cluster < 0) {
    const int64_t groups1 = (n_out + kCB - 1) / kCB;
    const int64_t cap2 = cluster_caps ? cluster_caps[1] : (int64_t)(num_sms / 2);
    if (groups1 <= cap2 && (K + kBK - 1) / kBK >= 2) nb = 1;
  }
  // Up projection above 32 MB of weights, up to 8 rows: units of four
  // 64-column blocks, i.e. 512-byte runs of every weight row (1 KB with
  // packed weights).  Measured with 2 GiB of weights rotating, d = 4096,
  // packed weights, calls back to back: M = 1 / 4 / 8 / 16: 37.0 / 37.2 /
  // 37.6 / 39.4 us against 37.0 / 37.2 / 38.5 / 38.9 with two blocks.  (Four
  // blocks issue twice the prefetches per unit; before an epilogue warp
  // issued them, M = 8 measured 38.7 against 38.6.)  Both layouts keep one
  // rule, so that swiglu_workspace_bytes serves both.
  if (!plain && !fp8 && tn.sk_nb < 0 && weight_bytes > kSkinnyClusterMaxWeightBytes && M <= 8)
    nb = 4;
  while (nb > 1 && nb * n > 256) nb /= 2;
  // FP8 down projection ([n_out, K] codes) above 32 MB of weights: two
  // 64-deep k blocks of one column block per unit, so every weight row is
  // read 256 contiguous bytes at a time instead of 128 (SWIGLU_SK_KB forces
  // 1 or 2).  Measured with 2 GiB of weights rotating, d = 4096: in 4-CTA
  // clusters M = 16 / 64 take 16.5 / 18.9 us against 17.7 / 20.4; in
  // stream-K mode, with the 384 KB prefetch below, M = 1 / 4 / 8 / 12 take
  // 15.0 / 15.2 / 15.5 / 15.6 us against 15.5 / 15.8 / 16.0 / 17.8.  The FP8
  // up projection measured slower this way (M = 1 / 16: 26.1 / 27.5 against
  // 24.1 / 25.9 us).
  p.kb = 1;
  const bool kb2 = tn.sk_kb >= 0 ? tn.sk_kb == 2
                                 : (plain && fp8 && weight_bytes > kSkinnyClusterMaxWeightBytes);
  if (fp8 && n <= 64 && kb2) {
    p.kb = 2;
    nb = 1;
  }
  p.nb = nb;
  p.l2_promo = tn.sk_promo >= 0 ? tn.sk_promo : 128;
  p.hint = tn.sk_hint >= 0 ? tn.sk_hint : 1;
  // Bulk-staged final sums (measured, calls back to back): the down
  // projection from M = 16 gains 1-4 % (d = 4096, M = 16: 25.5 -> 24.8 us;
  // M = 128: 44.4 -> 42.4 us; d = 8192, M = 32: 82.1 -> 80.1 us); at
  // M <= 8 and for the up projection, whose final sums are short, it is
  // within noise or up to 3 % slower.
  p.bulk = tn.sk_bulk >= 0 ? (tn.sk_bulk != 0) : (plain && M >= 16);
  // L2 prefetch budget per CTA, issued by an epilogue warp (measured, calls
  // back to back, 2 GiB of weights rotating, d = 4096):
  // - up projection: 512 KB with four-block units (packed, M = 1 / 4: 36.9
  //   / 36.9 us against 37.4 / 37.3 at 384 KB and 38.9 / 39.4 at 1 MB; M = 8:
  //   37.6 against 38.0 at 768 KB), 384 KB with two-block units (M = 16: 38.7
  //   against 39.1 at 512 KB); FP8: 512 KB (M = 1 / 16: 23.8 / 25.7 us
  //   against 24.9 / 26.0 at 768 KB).
  // - down projection with 256-column groups, whose sum kernel releases the
  //   next GEMM early (launch_skinny): 512 KB for bf16 (M = 1 / 16 / 48:
  //   20.9 / 21.5 / 23.7 us against 22.0 / 22.9 / 25.7 at 384 KB; the 256 KB
  //   of the one-kernel form, without the early release: 22.6 / 22.8 / 26.2),
  //   384 KB above 64 rows (M = 96 / 128: 23.7 / 24.7 us against 24.2 / 25.8
  //   at 512 KB), 384 KB for FP8 with one k block per unit (M = 1 / 8: 15.6
  //   / 16.2 against 15.9 / 16.4 at 256 KB);
  //   64 KB with the 128-column groups of larger M (M = 96 / 128 / 256: 26.9
  //   / 27.1 / 32.3 us against 28.7 / 29.0 / 34.0 at 256 KB; FP8 M = 256:
  //   26.9 against 28.1).
  // - FP8 down projection with units of two k blocks (stream-K, or 4-CTA
  //   clusters): 384 KB too (clusters, M = 16 / 32 / 64: 15.8 / 16.8 / 18.5
  //   us against 16.3 / 17.2 / 18.6 without; 64 or 128 KB measured slower
  //   than none, and all 448 KB of a CTA's range no faster).
  uint32_t pf_bytes = kPrefetchBytes;
  if (plain)
    pf_bytes = nb == 1 ? kPrefetchBytes / 8
                       : (fp8 || M > 64 ? kPrefetchBytes / 4 * 3 : kPrefetchBytes);
  else if (!fp8 && nb < 4)
    pf_bytes = kPrefetchBytes / 4 * 3;
  if (plain && fp8 && p.kb == 2) pf_bytes = kPrefetchBytes / 4 * 3;
  p.prefetch_units = tn.sk_prefetch_units >= 0 ? tn.sk_prefetch_units
                                               : (int)(pf_bytes / ((uint32_t)(nb * p.kb) * kSubBytes));
  const int64_t sub_cols = plain ? 2 * kCB : kCB;
  const int64_t subs = (n_out + sub_cols - 1) / sub_cols;
  p.n_cb = (subs + nb - 1) / nb;
  p.n_kb = (K + kBK * p.kb - 1) / (kBK * p.kb);
  p.units = p.n_cb * p.n_kb;
  p.grid = (int)(p.units < num_sms ? p.units : num_sms);
  if (p.grid < 1) p.grid = 1;
  // Cluster mode (measured): it wins when the weights are small enough that
  // the call is latency-bound (<= 32 MB), with the largest cluster size S
  // (<= 8, <= n_kb) whose n_cb clusters all run at once (cluster_caps[log2 S]
  // clusters of S fit on the GPU: 76 / 36 / 15 for S = 2 / 4 / 8 on GB300;
  // planning without a device assumes the same fractions of num_sms / S,
  // 1, 0.95 and 0.8, as clusters of 4 and 8 must fit whole GPCs).  d = 896: up projection in
  // 2-CTA clusters 8.3 us vs 9.2 us stream-K (4-CTA clusters, which need a
  // second wave, 12.8 us), 7.0 vs 12.5 us inside a CUDA graph (no workspace
  // to allocate and clear); down projection in 8-CTA clusters 8.6 vs 11.8 us.
  // With large weights stream-K is as fast or faster.  SWIGLU_SK_CLUSTER
  // overrides (0 = stream-K, 1/2/4/8 = that cluster size).
  int S = 1;
  for (int s = 8; s >= 2; s /= 2) {
    const int lg = s == 8 ? 3 : (s == 4 ? 2 : 1);
    const int64_t cap = cluster_caps ? cluster_caps[lg]
                                     : (int64_t)(num_sms / s * (s == 2 ? 1.0 : s == 4 ? 0.95 : 0.8));
    if (s <= p.n_kb && p.n_cb <= cap) {
      S = s;
      break;
    }
  }
  p.cluster = (S >= 2 && weight_bytes <= kSkinnyClusterMaxWeightBytes) ? S : 0;
  if (plain_cluster4) p.cluster = 4;
  const int forced = tn.sk_cluster;
  if (forced == 0) p.cluster = 0;
  if (forced == 1 || forced == 2 || forced == 4 || forced == 8)
    p.cluster = p.n_kb >= forced ? forced : 0;
  if (p.cluster) p.grid = (int)(p.n_cb * p.cluster);
  // Cluster mode (small weights): no L2 prefetch before the dependency wait
  // (measured, graph replay, d = 896: up projection M = 16 / 64: 6.9 / 8.1 us
  // with or without it; down projection M = 1 / 16 / 64: 6.8 / 7.2 / 8.0 us
  // without, 6.9 / 7.3 / 8.2 with 64 KB).  The FP8 down projection's 4-CTA
  // clusters keep their budget (above).
  if (p.cluster && !plain_cluster4 && tn.sk_prefetch_units < 0) p.prefetch_units = 0;
  const int64_t per = p.units > 0 ? p.units / p.grid : 1;   // fewest units a CTA gets
  p.maxq = (int)((p.n_kb + per - 1) / (per > 0 ? per : 1) + 1);
  p.counters_bytes = ((size_t)p.n_cb * sizeof(unsigned) + 255) / 256 * 256;
  p.part_bytes = (size_t)p.n_cb * p.maxq * nb * 2 * (size_t)M * kCB * sizeof(float);
  p.part_bytes = (p.part_bytes + 255) / 256 * 256;
  if (p.cluster) p.counters_bytes = p.part_bytes = 0;   // the reduction stays on chip
  // Two-kernel form (stream-K only; skinny_sum_kernel).  Measured, calls back
  // to back, one kernel / two kernels: the bf16 down projection d = 4096 at
  // M = 1 / 8 / 16: 21.9 / 22.9 / 25.2 us against 20.7 / 20.7 / 20.9 us;
  // d = 8192 at M = 16 / 128 / 256: 73.8 / 93.8 / 119.9 against 70.7 / 83.3
  // / 100.7 us; FP8, d = 4096, M = 1 / 8 / 256: 16.9 / 17.0 / 28.3 against
  // 16.9 / 18.0 / 60.5 us.  Where the group sums are short it loses the
  // second launch's cost: the up projection (d = 4096, M = 1: 35.9 against
  // 37.1 us).
  const bool split_default = plain;
  p.split = !p.cluster && (tn.sk_split >= 0 ? tn.sk_split > 0 : split_default) ? 1 : 0;
  return p;
}

cudaError_t skinny_cluster_caps(int caps[4]) {
  using C = SkCfg<16, 2>;
  auto kern = skinny_tc_kernel<16, 2, kSwiGLU, false, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::kSmemBytes);
  if (e != cudaSuccess) return e;
  caps[0] = 0;
  for (int lg = 1; lg <= 3; ++lg) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1u << lg;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1u << lg);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaOccupancyMaxActiveClusters(&caps[lg], kern, &cfg)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_skinny_tc(const void* x, const void* wa, const void* wb, void* out,
                             const void* resid, int64_t M, int64_t K, int64_t n_out,
                             int wlayout, const SkinnyPlan& p, float* part,
                             unsigned* counters, bool counters_clean, unsigned* status,
                             uint64_t timeout_ns, cudaStream_t st, const Fp8Scales* fp8) {
  if (p.units == 0 || M == 0) return cudaSuccess;
  if (fp8 && wlayout != kWeightsNK) return cudaErrorInvalidValue;
  CUtensorMap mx, mg, mu;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&mx, x, M, K, kBK, p.n_pad)) != cudaSuccess) return e;
  // weights as [K, n_out] (boxes 64 columns x 64 k) or [n_out, K] (64 k x 64 rows)
  const bool w_kmajor = wlayout == kWeightsNK, packed = wlayout == kWeightsPacked;
  if (packed && p.plain) return cudaErrorInvalidValue;
  const int64_t wr = w_kmajor ? n_out : K;
  const int64_t wc = w_kmajor ? K : (packed ? packed_cols(n_out) : n_out);
  if ((e = make_tmap_bf16_2d(&mg, wa, wr, wc, 64, 64, p.l2_promo)) != cudaSuccess) return e;
  if (p.plain || packed) {
    mu = mg;
  } else if ((e = make_tmap_bf16_2d(&mu, wb, wr, wc, 64, 64, p.l2_promo)) != cudaSuccess) {
    return e;
  }
  // Arrival counters must be zero on entry (stream-K mode only).
  if (!p.cluster && !counters_clean &&
      (e = cudaMemsetAsync(counters, 0, (size_t)p.n_cb * sizeof(unsigned), st)) != cudaSuccess)
    return e;
  SkArgs a;
  a.M = (int)M;
  a.n_out = (int)n_out;
  a.n_kb = (int)p.n_kb;
  a.maxq = p.maxq;
  a.units = p.units;
  a.grid = p.grid;
  a.hint = p.hint;
  a.kmajor = w_kmajor ? 1 : 0;
  a.packed = packed ? 1 : 0;
  a.sx = fp8 ? fp8->sx : nullptr;
  a.sw_a = fp8 ? fp8->sw_a : nullptr;
  a.sw_b = fp8 ? fp8->sw_b : nullptr;
  a.prefetch_units = p.prefetch_units;
  a.bulk = p.bulk;
  a.split = p.split;
  a.nb = p.nb;
  // The sum kernel releases the next kernel before its own wait for FP8
  // calls (the next one starts with the activation quantizer) and for the
  // down projection's 256-column groups, whose next GEMM then prefetches 512
  // KB while this call's sums run (see plan_skinny's prefetch budgets).
  a.release_early = (fp8 || (p.plain && p.nb >= 2)) ? 1 : 0;
  a.k64 = (int)((K + kBK - 1) / kBK);
  a.cluster = p.cluster;
  a.part = part;
  a.counters = counters;
  a.out = (uint16_t*)out;
  a.resid = (const uint16_t*)resid;
  a.status = status;
  a.timeout_ns = timeout_ns;
  if (p.plain)
    e = fp8 ? launch_mode<kPlain, true>(p.n_pad, p.nb, p.kb, mx, mg, mu, a, st)
            : launch_mode<kPlain, false>(p.n_pad, p.nb, p.kb, mx, mg, mu, a, st);
  else
    e = fp8 ? launch_mode<kSwiGLU, true>(p.n_pad, p.nb, p.kb, mx, mg, mu, a, st)
            : launch_mode<kSwiGLU, false>(p.n_pad, p.nb, p.kb, mx, mg, mu, a, st);
  if (e != cudaSuccess || !a.split) return e;
  if (p.plain) return fp8 ? launch_sum<kPlain, true>(a, st) : launch_sum<kPlain, false>(a, st);
  return fp8 ? launch_sum<kSwiGLU, true>(a, st) : launch_sum<kSwiGLU, false>(a, st);
}

}  // namespace swg
