// S1 (SIMT): split-K partial sums of x.W_gate and x.W_up on the CUDA cores.
//
// Follows the skinny-matrix kernel of "Ou part le temps d'un token", section
// "Un kernel pour les matrices etroites": the grid is cut along the weights
// (which are large), not along the output (which is small).  A CTA of 8 warps
// owns one block of adjacent weight columns and one slice of the shared
// dimension K; lane l of every warp reads the same 16 contiguous bytes of a
// weight row (a warp covers 512 contiguous bytes, fully coalesced), and warp w
// takes every 8th k of the slice.  Each thread keeps 4 k-rows of both
// matrices in flight before using them.  The 8 warp sums are combined through
// shared memory in warp order, and each slice writes its partial sum; the
// slices are then added in slice order, so the result does not depend on CTA
// scheduling.  That sum and the SwiGLU epilogue run either in the reduction
// kernel (reduce_swiglu.cu) or, in the single-launch form, in this kernel:
// the last CTA of a column block to finish (an atomic ticket; nothing waits)
// adds the slices, exactly as the reduction kernel does, and stores h.  The
// page's "Ce qui reste : les lancements" finds the second launch to be a
// large part of a small product's time.
//
// Differences from the page's design, for GB300: 16-byte loads (4 f32 or
// 8 bf16 per lane instead of one f32), both weight matrices streamed by the
// same CTA (one pass over x for gate and up), up to 4 rows of x per CTA, and
// the slice target scaled to this GPU's SM count.  This path serves f32 (all
// M) and is the CUDA-core reference path for bf16; the tensor-core paths
// serve bf16 by default.
#include <atomic>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kUnroll = 4;          // k rows in flight per thread per matrix
constexpr int kMaxKPerSlice = 1024; // bounds the staged slice of x
constexpr int kMinKPerSlice = 64;   // minimum slice depth ("Ou part le temps d'un token", "Un kernel pour les matrices etroites")
constexpr int kCtasPerSmTarget = 4;

template <bool BF16>
__device__ __forceinline__ void unpack16(const uint4& v, float* f) {
  if constexpr (BF16) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  } else {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
}

// counters == null: write the partial sums only.  Otherwise (single launch)
// counters holds one arrival counter per (column block, row chunk), zero on
// entry and left at zero, and the last CTA of each writes h.
template <bool BF16, int RC>
__global__ void __launch_bounds__(kThreads)
simt_partial_kernel(const void* __restrict__ x_, const void* __restrict__ wg_,
                    const void* __restrict__ wu_, float* __restrict__ part,
                    int M, int d, int d_ff, int ks, unsigned* __restrict__ counters,
                    void* __restrict__ h, int packed) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int C = 32 * VEC;
  constexpr int ES = BF16 ? 2 : 4;
  extern __shared__ float smem[];  // x slice [RC][kn], then warp sums [8][RC][2][C]

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int s = blockIdx.y;
  const int row0 = blockIdx.z * RC;
  const int k0 = s * ks;
  const int k1 = min(d, k0 + ks);
  const int kn = k1 - k0;
  const int col = blockIdx.x * C + lane * VEC;
  const bool valid = col < d_ff;
  // Launched with programmatic stream serialisation: wait for the previous
  // kernel before touching x or the partial-sum buffer, then let the
  // reduction kernel be scheduled.
  tc::pdl_wait();
  tc::pdl_launch_dependents();

  // Stage x[row0 : row0+RC, k0 : k1] in shared memory as f32 (rows past M are 0).
  for (int t = threadIdx.x; t < RC * kn; t += kThreads) {
    const int r = t / kn, k = t - r * kn, row = row0 + r;
    float v = 0.f;
    if (row < M) {
      const size_t idx = (size_t)row * d + k0 + k;
      if constexpr (BF16)
        v = bf16_lo(((const uint16_t*)x_)[idx]);
      else
        v = ((const float*)x_)[idx];
    }
    smem[r * kn + k] = v;
  }
  __syncthreads();

  float accg[RC][VEC], accu[RC][VEC];
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int v = 0; v < VEC; ++v) accg[r][v] = accu[r][v] = 0.f;

  if (valid) {
    // packed weights: gate block b of 64 columns at packed column 128 b, up at
    // 128 b + 64 (a lane's VEC columns never straddle a block)
    const int gcol = packed ? col + (col & ~63) : col;
    const int ucol = packed ? gcol + 64 : col;
    const char* wg = (const char*)wg_ + (size_t)gcol * ES;
    const char* wu = (const char*)wu_ + (size_t)ucol * ES;
    const size_t row_bytes = (size_t)(packed ? 128 * ((d_ff + 63) / 64) : d_ff) * ES;
    for (int k = k0 + warp; k < k1; k += kWarps * kUnroll) {
      uint4 vg[kUnroll], vu[kUnroll];
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int kk = k + q * kWarps;
        if (kk < k1) {
          vg[q] = ldg_stream_v4(wg + (size_t)kk * row_bytes);
          vu[q] = ldg_stream_v4(wu + (size_t)kk * row_bytes);
        }
      }
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int kk = k + q * kWarps;
        if (kk < k1) {
          float fg[VEC], fu[VEC];
          unpack16<BF16>(vg[q], fg);
          unpack16<BF16>(vu[q], fu);
#pragma unroll
          for (int r = 0; r < RC; ++r) {
            const float xv = smem[r * kn + (kk - k0)];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              accg[r][v] = fmaf(xv, fg[v], accg[r][v]);
              accu[r][v] = fmaf(xv, fu[v], accu[r][v]);
            }
          }
        }
      }
    }
  }
  __syncthreads();  // the x slice is no longer needed; reuse the buffer

  float* red = smem;
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      red[((warp * RC + r) * 2 + 0) * C + lane * VEC + v] = accg[r][v];
      red[((warp * RC + r) * 2 + 1) * C + lane * VEC + v] = accu[r][v];
    }
  __syncthreads();

  // Sum the 8 warps in warp order and write this slice's partial sums.
  for (int t = threadIdx.x; t < RC * 2 * C; t += kThreads) {
    const int c = t % C, gu = (t / C) & 1, r = t / (2 * C);
    const int row = row0 + r, j = blockIdx.x * C + c;
    if (row < M && j < d_ff) {
      float sum = red[((0 * RC + r) * 2 + gu) * C + c];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) sum += red[((w * RC + r) * 2 + gu) * C + c];
      part[(((size_t)s * M + row) * 2 + gu) * d_ff + j] = sum;
    }
  }
  if (!counters) return;

  // Single launch: the last slice of this column block and row chunk to
  // arrive sums the slices in slice order and applies the epilogue.
  __shared__ unsigned ticket;
  __threadfence();
  __syncthreads();
  unsigned* ctr = counters + (size_t)blockIdx.z * gridDim.x + blockIdx.x;
  if (threadIdx.x == 0) ticket = atomicAdd(ctr, 1u);
  __syncthreads();
  if (ticket + 1u != gridDim.y) return;
  __threadfence();
  // one thread = 4 adjacent outputs of one row (d_ff is a multiple of 4),
  // the same sums and rounding as the reduction kernel
  for (int t = threadIdx.x; t < RC * (C / 4); t += kThreads) {
    const int r = t / (C / 4), row = row0 + r;
    const int j = blockIdx.x * C + (t - r * (C / 4)) * 4;
    if (row >= M || j >= d_ff) continue;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int q = 0; q < (int)gridDim.y; ++q) {
      const float* pg = part + (((size_t)q * M + row) * 2) * d_ff + j;
      const float4 a = __ldcg(reinterpret_cast<const float4*>(pg));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(pg + d_ff));
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
    }
    if constexpr (BF16) {
      uint2 o;
      o.x = pack_bf16x2(silu_fast(g.x) * u.x, silu_fast(g.y) * u.y);
      o.y = pack_bf16x2(silu_fast(g.z) * u.z, silu_fast(g.w) * u.w);
      *reinterpret_cast<uint2*>((uint16_t*)h + (size_t)row * d_ff + j) = o;
    } else {
      *reinterpret_cast<float4*>((float*)h + (size_t)row * d_ff + j) =
          make_float4(silu_accurate(g.x) * u.x, silu_accurate(g.y) * u.y,
                      silu_accurate(g.z) * u.z, silu_accurate(g.w) * u.w);
    }
  }
  if (threadIdx.x == 0) *ctr = 0u;   // left at zero for the next call
}

template <bool BF16, int RC>
cudaError_t launch_one(const void* x, const void* wg, const void* wu, float* part,
                       int64_t M, int64_t d, int64_t d_ff, const SimtPlan& p,
                       unsigned* counters, void* h, bool packed, cudaStream_t st) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int C = 32 * VEC;
  const size_t x_bytes = (size_t)RC * p.k_per_slice * sizeof(float);
  const size_t red_bytes = (size_t)kWarps * RC * 2 * C * sizeof(float);
  const size_t smem = x_bytes > red_bytes ? x_bytes : red_bytes;
  auto kern = simt_partial_kernel<BF16, RC>;
  // The opt-in shared-memory limit is a per-function, per-device attribute:
  // set it once per device to the largest size this instantiation can use.
  static std::atomic<int> configured[64];   // zero: not yet set on that device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    const size_t most = (size_t)RC * kMaxKPerSlice * sizeof(float) > red_bytes
                            ? (size_t)RC * kMaxKPerSlice * sizeof(float) : red_bytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(1, std::memory_order_release);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.col_blocks, (unsigned)p.slices, (unsigned)p.row_chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, x, wg, wu, part, (int)M, (int)d, (int)d_ff,
                            (int)p.k_per_slice, counters, h, packed ? 1 : 0);
}

}  // namespace

int64_t split_k_slices(int64_t K, int64_t col_blocks, int64_t target_blocks,
                       int64_t min_k_per_slice);

SimtPlan plan_simt(int64_t M, int64_t d, int64_t d_ff, int dtype, int num_sms,
                   const Tuning& tn) {
  SimtPlan p{};
  p.vec = dtype == 1 ? 8 : 4;
  p.cols_per_cta = 32 * p.vec;
  p.row_chunk = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
  p.col_blocks = (d_ff + p.cols_per_cta - 1) / p.cols_per_cta;
  p.row_chunks = (M + p.row_chunk - 1) / p.row_chunk;
  if (d <= 0 || M <= 0 || d_ff <= 0) {
    p.slices = 0;
    p.k_per_slice = 0;
    return p;
  }
  int64_t s = split_k_slices(d, p.col_blocks * p.row_chunks,
                             (int64_t)kCtasPerSmTarget * num_sms, kMinKPerSlice);
  const int64_t s_min = (d + kMaxKPerSlice - 1) / kMaxKPerSlice;
  if (s < s_min) s = s_min;
  int64_t ks = (d + s - 1) / s;
  ks = (ks + 7) / 8 * 8;
  p.k_per_slice = ks;
  p.slices = (d + ks - 1) / ks;
  // Single launch wherever the arrival counters fit the per-stream counter
  // region (every decode shape); SWIGLU_SIMT_FUSED = 0 keeps two launches.
  const int64_t n_ctr = p.col_blocks * p.row_chunks;
  p.fused = tn.simt_fused != 0 && n_ctr * (int64_t)sizeof(unsigned) <= (int64_t)kStreamCounterBytes;
  p.counters_bytes = p.fused ? ((size_t)n_ctr * sizeof(unsigned) + 255) / 256 * 256 : 0;
  return p;
}

cudaError_t launch_simt_partial(const void* x, const void* wg, const void* wu,
                                float* part, int64_t M, int64_t d, int64_t d_ff,
                                int dtype, const SimtPlan& p, cudaStream_t st,
                                unsigned* counters, bool counters_clean, void* h,
                                bool packed) {
  if (p.slices == 0) return cudaSuccess;
  if (counters && !counters_clean) {
    cudaError_t e = cudaMemsetAsync(counters, 0, p.counters_bytes, st);
    if (e != cudaSuccess) return e;
  }
  if (!counters) h = nullptr;
  const bool bf16 = dtype == 1;
  switch (p.row_chunk) {
    case 1: return bf16 ? launch_one<true, 1>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st)
                        : launch_one<false, 1>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st);
    case 2: return bf16 ? launch_one<true, 2>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st)
                        : launch_one<false, 2>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st);
    default: return bf16 ? launch_one<true, 4>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st)
                         : launch_one<false, 4>(x, wg, wu, part, M, d, d_ff, p, counters, h, packed, st);
  }
}

}  // namespace swg
