// S2: fixed-order reduction of the split-K partial sums, then the SwiGLU
// epilogue h = silu(g) * u, rounded once to the output type.
//
// "Ou part le temps d'un token", section "Un kernel pour les matrices
// etroites": each slice writes its partial sum and a second kernel adds them,
// in an order that does not depend on which CTA finished first (atomics in
// the output would change the result by a few ulps from run to run).  The
// section "Deux operations de trop" puts the bias of an affine layer into
// this same reduction pass; here the pass carries the activation instead, so
// g and u exist only as f32 partials and are combined only once complete.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {

namespace {

constexpr int kThreads = 256;

template <bool BF16>
__global__ void __launch_bounds__(kThreads)
reduce_swiglu_kernel(const float* __restrict__ part, void* __restrict__ h,
                     int64_t M, int64_t d_ff, int slices) {
  // Launched with programmatic stream serialisation behind the partial-sum
  // kernel: its launch overlaps that kernel, and it reads the partial sums
  // only once that kernel has finished and its writes are visible.
  tc::pdl_wait();
  tc::pdl_launch_dependents();
  // One thread = 4 adjacent outputs of one row (d_ff is a multiple of 4).
  const int64_t groups = d_ff >> 2;
  const int64_t total = M * groups;
  for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * kThreads) {
    const int64_t m = t / groups;
    const int64_t j = (t - m * groups) << 2;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int s = 0; s < slices; ++s) {
      const float* pg = part + (((int64_t)s * M + m) * 2) * d_ff + j;
      const float4 a = __ldcg(reinterpret_cast<const float4*>(pg));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(pg + d_ff));
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
    }
    float r0, r1, r2, r3;
    if constexpr (BF16) {
      r0 = silu_fast(g.x) * u.x; r1 = silu_fast(g.y) * u.y;
      r2 = silu_fast(g.z) * u.z; r3 = silu_fast(g.w) * u.w;
      uint2 o;
      o.x = pack_bf16x2(r0, r1);
      o.y = pack_bf16x2(r2, r3);
      *reinterpret_cast<uint2*>((uint16_t*)h + m * d_ff + j) = o;
    } else {
      r0 = silu_accurate(g.x) * u.x; r1 = silu_accurate(g.y) * u.y;
      r2 = silu_accurate(g.z) * u.z; r3 = silu_accurate(g.w) * u.w;
      *reinterpret_cast<float4*>((float*)h + m * d_ff + j) = make_float4(r0, r1, r2, r3);
    }
  }
}

}  // namespace

cudaError_t launch_reduce_swiglu(const float* part, void* h, int64_t M,
                                 int64_t d_ff, int64_t slices, int dtype,
                                 int num_sms, cudaStream_t st) {
  const int64_t total = M * (d_ff >> 2);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms * 16;
  if (blocks > cap) blocks = cap;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == 1)
    return cudaLaunchKernelEx(&cfg, reduce_swiglu_kernel<true>, part, h, M, d_ff, (int)slices);
  return cudaLaunchKernelEx(&cfg, reduce_swiglu_kernel<false>, part, h, M, d_ff, (int)slices);
}

}  // namespace swg
