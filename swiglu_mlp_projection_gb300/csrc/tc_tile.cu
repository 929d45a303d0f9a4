// Large-M path on the tensor cores (bf16): a persistent tcgen05 GEMM whose
// epilogue applies SwiGLU to the accumulator tile before one bf16 store.
//
// "Tile-Level Activation Overlap for Efficient LLM Inference" fuses SwiGLU
// into the GEMM at tile level so that neither Gate nor Up is ever written to
// HBM; its Kernel-2 interleaves the gate and up weight columns so one GEMM
// tile holds matching gate/up column pairs and its epilogue emits
// SiLU(gate) * up.  This kernel keeps that idea and re-does the rest for
// sm_103a:
//   * an output tile is 128 rows x 128 columns of h; its accumulator is
//     128 x 256 f32 in TMEM: columns 0-127 = x.W_gate, 128-255 = x.W_up for
//     the same 128 output columns (the interleave happens per 64-column TMA
//     box while loading; W_gate and W_up stay separate row-major arrays);
//   * A = x tile (K-major), B = the four weight boxes (MN-major, read straight
//     from the row-major weights), both TMA-staged in a 4-stage ring;
//   * one thread issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM
//     accumulators, so the epilogue of tile i overlaps the MMAs of tile i+1
//     (the overlap the paper gets from ping-pong warp groups);
//   * the epilogue (4 warps, one accumulator row per thread) reads gate and up
//     columns with tcgen05.ld, computes silu(g) * u in f32, rounds to bf16 into
//     a 128-byte-swizzled staging tile and TMA-stores it.
// Tiles are visited column-block-major so the CTAs running at the same time
// share weight columns and x rows through L2.
//
// In its plain mode the same kernel computes the down projection
// y = h . W_down (+ residual) ("1 . Anatomie d'un transformeur sur GPU",
// section 1.6, kernels #10 and #11): the 256 accumulator columns are 256
// adjacent output columns, and the epilogue adds the residual and stores
// them in two 128-column passes.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {
namespace {

using namespace tc;

constexpr int kBM = 128;                        // output rows per tile
constexpr int kBN = 128;                        // output columns per tile
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kChunkBytes = 64 * kBK * 2;  // 8 KB: one 64-column weight box
constexpr uint32_t kBBytes = 4 * kChunkBytes;   // gate 0-63, gate 64-127, up 0-63, up 64-127
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kStagingHalf = kBM * 128;    // 128 rows x 64 bf16
constexpr uint32_t kStagingBytes = 2 * kStagingHalf;
constexpr uint32_t kTmemCols = 512;             // two 128 x 256 f32 accumulators
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kStagingBytes + 256;

struct TileArgs {
  int n_mb, n_nb, n_kb, n_out;   // n_out: output columns
  int M;
  int64_t tiles;
  const uint16_t* resid;         // plain mode: [M][n_out] added to the sums, or null
  int kmajor;                    // weights stored [n_out, K] instead of [K, n_out]
  unsigned* status;
  uint64_t timeout_ns;
};

constexpr int kSwiGLU = 0;       // accumulator = 128 gate columns | 128 up columns
constexpr int kPlain = 1;        // accumulator = 256 adjacent output columns

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, unsigned* status,
                                           uint64_t timeout_ns) {
  int never = 0;
  return mbar_wait(bar, parity, &never, status, timeout_ns);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
tile_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
               const __grid_constant__ CUtensorMap tm_wu, const __grid_constant__ CUtensorMap tm_h,
               const TileArgs a) {
  // output columns per tile, and where the four 64-column B boxes come from
  constexpr int kOutCols = MODE == kSwiGLU ? kBN : 2 * kBN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint8_t* staging = stages + (size_t)kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStagingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], kEpiThreads);
    mbar_init(&tempty[1], kEpiThreads);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
    tma_prefetch_desc(&tm_h);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The set-up above overlaps the previous kernel's tail; x and h are touched
  // only after it has finished.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < a.tiles; t += gridDim.x) {
        const int mb = (int)(t % a.n_mb), nb = (int)(t / a.n_mb);
        for (int kb = 0; kb < a.n_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)stage * kStageBytes;
          uint8_t* sb = st + kABytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tma_load_2d(st, &tm_x, &full[stage], kb * kBK, mb * kBM);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // box q of the B tile: SwiGLU -> gate 0-63, gate 64-127, up 0-63,
            // up 64-127 of this tile's columns; plain -> 4 x 64 adjacent columns
            const CUtensorMap* m = (MODE == kSwiGLU && q >= 2) ? &tm_wu : &tm_wg;
            const int col = MODE == kSwiGLU ? nb * kBN + 64 * (q & 1) : nb * kOutCols + 64 * q;
            if (a.kmajor)
              tma_load_2d(sb + q * kChunkBytes, m, &full[stage], kb * kBK, col);
            else
              tma_load_2d(sb + q * kChunkBytes, m, &full[stage], col, kb * kBK);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        const int64_t first = issued > kStages ? issued - kStages : 0;
        for (int64_t i = first; i < issued; ++i)
          wait_drain(&full[i % kStages], (uint32_t)((i / kStages) & 1), a.status, a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // A (x) is K-major; B (the weights) MN-major for [K, n_out] weights,
      // K-major for [n_out, K] weights.
      const uint32_t idesc = a.kmajor ? idesc_bf16_f32(kBM, 2 * kBN, false, false)
                                      : idesc_bf16_f32(kBM, 2 * kBN, false, true);
      const uint32_t b_step = a.kmajor ? 32u : 2048u;
      const uint32_t b_lbo = a.kmajor ? 16u : kChunkBytes;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < a.tiles; t += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * 2 * kBN);
        for (int kb = 0; kb < a.n_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + (size_t)stage * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32u, 16u, 1024u);
            const uint64_t bd = smem_desc_sw128(b_addr + kk * b_step, b_lbo, 1024u);
            mma_bf16(d_tmem, ad, bd, idesc, (kb != 0 || kk != 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == kStages) {
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
      }
      mma_commit(drain);
      wait_drain(drain, 0, a.status, a.timeout_ns);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // accumulator row = output row in the tile
    const int et = threadIdx.x - 64;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    constexpr int kPasses = MODE == kSwiGLU ? 1 : 2;   // 128 output columns per pass
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < a.tiles; t += gridDim.x) {
      const int mb = (int)(t % a.n_mb), nb = (int)(t / a.n_mb);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, a.status, a.timeout_ns)) break;
      tc_fence_after();
      const int64_t grow = (int64_t)mb * kBM + row;       // output row of this thread
      for (int pass = 0; pass < kPasses; ++pass) {
        if (et == 0) bulk_wait_read0();   // the previous store has read the staging tile
        __syncwarp();
        named_bar_sync(1, kEpiThreads);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t g[32], u[32];
          const uint32_t col0 = (uint32_t)(acc * 2 * kBN + pass * kBN + ch * 32);
          tmem_ld_x32(tmem + lane_off + col0, g);
          if constexpr (MODE == kSwiGLU) tmem_ld_x32(tmem + lane_off + col0 + kBN, u);
          tmem_wait_ld();
          float rv[32];
          if constexpr (MODE == kPlain) {
            // residual row segment: 32 bf16 of this output row
            const int64_t c0 = (int64_t)nb * kOutCols + pass * kBN + ch * 32;
            const bool has = a.resid && grow < a.M && c0 < a.n_out;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w = make_uint4(0u, 0u, 0u, 0u);
              if (has && c0 + 8 * v < a.n_out)
                w = *reinterpret_cast<const uint4*>(a.resid + grow * a.n_out + c0 + 8 * v);
              rv[8 * v + 0] = bf16_lo(w.x); rv[8 * v + 1] = bf16_hi(w.x);
              rv[8 * v + 2] = bf16_lo(w.y); rv[8 * v + 3] = bf16_hi(w.y);
              rv[8 * v + 4] = bf16_lo(w.z); rv[8 * v + 5] = bf16_hi(w.z);
              rv[8 * v + 6] = bf16_lo(w.w); rv[8 * v + 7] = bf16_hi(w.w);
            }
          }
          uint8_t* rowp = staging + (ch >> 1) * kStagingHalf + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 8 * i + 2 * e;
              float o0, o1;
              if constexpr (MODE == kSwiGLU) {
                o0 = silu_fast(__uint_as_float(g[q])) * __uint_as_float(u[q]);
                o1 = silu_fast(__uint_as_float(g[q + 1])) * __uint_as_float(u[q + 1]);
              } else {
                o0 = __uint_as_float(g[q]) + rv[q];
                o1 = __uint_as_float(g[q + 1]) + rv[q + 1];
              }
              w[e] = pack_bf16x2(o0, o1);
            }
            const int chunk = ((ch & 1) * 4 + i) ^ (row & 7);   // 128-byte swizzle
            *reinterpret_cast<uint4*>(rowp + chunk * 16) = v;
          }
        }
        if (pass == kPasses - 1) {
          // every accumulator column of this buffer has been read
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
        }
        fence_async_smem();
        __syncwarp();
        named_bar_sync(1, kEpiThreads);
        if (et == 0) {
          const int c0 = nb * kOutCols + pass * kBN;
          if (c0 < a.n_out) tma_store_2d(&tm_h, staging, c0, mb * kBM);
          if (c0 + 64 < a.n_out) tma_store_2d(&tm_h, staging + kStagingHalf, c0 + 64, mb * kBM);
          bulk_commit();
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (et == 0) bulk_wait0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

TilePlan plan_tile(int64_t M, int64_t K, int64_t n_out, int num_sms, bool plain) {
  (void)K;
  TilePlan p{};
  const int64_t cols = plain ? 2 * kBN : kBN;
  p.plain = plain;
  p.n_mb = (M + kBM - 1) / kBM;
  p.n_nb = (n_out + cols - 1) / cols;
  p.tiles = p.n_mb * p.n_nb;
  p.grid = (int)(p.tiles < num_sms ? p.tiles : num_sms);
  if (p.grid < 1) p.grid = 1;
  return p;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mu,
                        const CUtensorMap& mh, const TileArgs& a, int grid, cudaStream_t st) {
  auto kern = tile_tc_kernel<MODE>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = 1;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mx, mg, mu, mh, a);
}

cudaError_t launch_tile_tc(const void* x, const void* wa, const void* wb, void* out,
                           const void* resid, int64_t M, int64_t K, int64_t n_out,
                           bool w_kmajor, const TilePlan& p, unsigned* status,
                           uint64_t timeout_ns, cudaStream_t st) {
  if (p.tiles == 0 || K == 0) return cudaSuccess;
  CUtensorMap mx, mg, mu, mh;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&mx, x, M, K, kBK, kBM)) != cudaSuccess) return e;
  const int64_t wr = w_kmajor ? n_out : K, wc = w_kmajor ? K : n_out;
  if ((e = make_tmap_bf16_2d(&mg, wa, wr, wc, 64, 64)) != cudaSuccess) return e;
  if (p.plain) {
    mu = mg;
  } else if ((e = make_tmap_bf16_2d(&mu, wb, wr, wc, 64, 64)) != cudaSuccess) {
    return e;
  }
  if ((e = make_tmap_bf16_2d(&mh, out, M, n_out, 64, kBM)) != cudaSuccess) return e;
  TileArgs a;
  a.n_mb = (int)p.n_mb;
  a.n_nb = (int)p.n_nb;
  a.n_kb = (int)((K + kBK - 1) / kBK);
  a.n_out = (int)n_out;
  a.M = (int)M;
  a.tiles = p.tiles;
  a.resid = (const uint16_t*)resid;
  a.kmajor = w_kmajor ? 1 : 0;
  a.status = status;
  a.timeout_ns = timeout_ns;
  return p.plain ? launch_mode<kPlain>(mx, mg, mu, mh, a, p.grid, st)
                 : launch_mode<kSwiGLU>(mx, mg, mu, mh, a, p.grid, st);
}

}  // namespace swg
