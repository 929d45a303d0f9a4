// FP8 (e4m3) quantization for the FP8 up projection: activations per row,
// weights per output column.
//
// A row (or column) with amax = max |v| gets the multiplier 448 / amax and
// the dequantization scale amax / 448 (both one f32 division; 448 is the
// largest finite e4m3 value); each element becomes the e4m3 code of the f32
// product v * (448 / amax), rounded to nearest even and saturated to +-448
// (cvt.rn.satfinite).  An all-zero row gets multiplier 0 and scale 0.  The
// FP8 kernels then compute sum_k x8 w8 in f32 on the tensor cores and apply
// sx[i] * sw[j] to each sum.
//
// Weights are quantized once (their codes are written [d_ff, d], the shared
// dimension contiguous, which is what tcgen05 reads for 8-bit operands);
// activations on every call, by a small kernel ahead of the GEMM.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {
namespace {

constexpr int kThreads = 256;

// Two f32 -> two e4m3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kThreads / 32 ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// Eight bf16 -> eight e4m3 codes of v * inv.
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  uint2 o;
  o.x = e4m3x2(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv) |
        (e4m3x2(bf16_lo(v.y) * inv, bf16_hi(v.y) * inv) << 16);
  o.y = e4m3x2(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv) |
        (e4m3x2(bf16_lo(v.w) * inv, bf16_hi(v.w) * inv) << 16);
  return o;
}

__device__ __forceinline__ float amax8(const uint4& v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
  return m;
}

// A row of up to kThreads * kRowItems groups of 8 values is held in registers:
// every load of the row is issued before any is used, and the codes are made
// from the same registers (K up to 16384 here).
constexpr int kRowItems = 8;

// One CTA per row of x [M, K] (bf16, K a multiple of 16): codes [M, K], scales [M].
__global__ void __launch_bounds__(kThreads)
quantize_rows_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ codes,
                     float* __restrict__ scales, int64_t K) {
  __shared__ float red[kThreads / 32];
  // Launched with programmatic serialisation: x may still be written by the
  // previous kernel, and the previous GEMM may still read codes / scales, so
  // everything waits.  The GEMM that follows may launch at once: it prefetches
  // its weights into L2 while the previous GEMM finishes, and its own
  // dependency wait covers this kernel (which completes only after the
  // previous one has).
  tc::pdl_launch_dependents();
  tc::pdl_wait();
  const int64_t r = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + r * K);
  uint2* dst = reinterpret_cast<uint2*>(codes + r * K);
  const int64_t n8 = K / 8;
  float amax = 0.f;
  if (n8 <= (int64_t)kThreads * kRowItems) {
    uint4 v[kRowItems];
#pragma unroll
    for (int j = 0; j < kRowItems; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * kThreads;
      if (i < n8) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < kRowItems; ++j)
      if (threadIdx.x + (int64_t)j * kThreads < n8) amax = amax8(v[j], amax);
    amax = block_max(amax, red);
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
#pragma unroll
    for (int j = 0; j < kRowItems; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * kThreads;
      if (i < n8) dst[i] = quant8(v[j], inv);
    }
  } else {
    for (int64_t i = threadIdx.x; i < n8; i += kThreads) amax = amax8(src[i], amax);
    amax = block_max(amax, red);
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
    for (int64_t i = threadIdx.x; i < n8; i += kThreads) dst[i] = quant8(src[i], inv);
  }
  if (threadIdx.x == 0) scales[r] = amax > 0.f ? amax / 448.0f : 0.f;
}

// Column amax of w [K, N] (bf16): CTA (blockIdx.x, blockIdx.y) covers 256
// columns and a range of rows; the maxima meet in amax_bits (f32 bits of
// non-negative values order like the values; zero on entry).
__global__ void __launch_bounds__(kThreads)
col_amax_kernel(const uint16_t* __restrict__ w, unsigned* __restrict__ amax_bits, int64_t K,
                int64_t N, int64_t rows_per_cta) {
  const int64_t j = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (j >= N) return;
  const int64_t k0 = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t k1 = k0 + rows_per_cta < K ? k0 + rows_per_cta : K;
  float m = 0.f;
  for (int64_t k = k0; k < k1; ++k) m = fmaxf(m, fabsf(bf16_lo(w[k * N + j])));
  atomicMax(amax_bits + j, __float_as_uint(m));
}

// Codes of w [K, N] by 64 x 64 tiles, written transposed: codes_nk [N, K].
// Also writes the scales (tile row 0 of each column block).
__global__ void __launch_bounds__(kThreads)
quantize_cols_kernel(const uint16_t* __restrict__ w, const unsigned* __restrict__ amax_bits,
                     uint8_t* __restrict__ codes_nk, float* __restrict__ scales, int64_t K,
                     int64_t N) {
  __shared__ float tile[64][65];
  const int64_t j0 = (int64_t)blockIdx.x * 64, k0 = (int64_t)blockIdx.y * 64;
  // load: 64 rows (k) x 64 columns (j), columns contiguous
  for (int t = threadIdx.x; t < 64 * 64; t += kThreads) {
    const int kk = t >> 6, jj = t & 63;
    const int64_t k = k0 + kk, j = j0 + jj;
    tile[kk][jj] = (k < K && j < N) ? bf16_lo(w[k * N + j]) : 0.f;
  }
  __syncthreads();
  // store: for each column j, 64 consecutive k as 32 code pairs
  for (int t = threadIdx.x; t < 64 * 32; t += kThreads) {
    const int jj = t >> 5, kp = (t & 31) * 2;
    const int64_t j = j0 + jj, k = k0 + kp;
    if (j >= N || k >= K) continue;
    const float amax = __uint_as_float(amax_bits[j]);
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
    const uint32_t c = e4m3x2(tile[kp][jj] * inv, tile[kp + 1][jj] * inv);
    *reinterpret_cast<uint16_t*>(codes_nk + j * K + k) = (uint16_t)c;
  }
  if (blockIdx.y == 0) {
    for (int jj = threadIdx.x; jj < 64; jj += kThreads) {
      const int64_t j = j0 + jj;
      if (j >= N) continue;
      const float amax = __uint_as_float(amax_bits[j]);
      scales[j] = amax > 0.f ? amax / 448.0f : 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows_fp8(const void* x, void* codes, float* scales, int64_t M,
                                     int64_t K, cudaStream_t st) {
  if (M == 0 || K == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_rows_kernel, (const uint16_t*)x, (uint8_t*)codes,
                            scales, K);
}

cudaError_t launch_quantize_cols_fp8(const void* w, void* codes_nk, float* scales,
                                     unsigned* amax_scratch, int64_t K, int64_t N,
                                     int num_sms, cudaStream_t st) {
  if (K == 0 || N == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(amax_scratch, 0, (size_t)N * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  const int64_t cblocks = (N + kThreads - 1) / kThreads;
  int64_t splits = ((int64_t)num_sms * 4 + cblocks - 1) / cblocks;
  if (splits > K) splits = K;
  if (splits < 1) splits = 1;
  const int64_t rows = (K + splits - 1) / splits;
  col_amax_kernel<<<dim3((unsigned)cblocks, (unsigned)((K + rows - 1) / rows)), kThreads, 0,
                    st>>>((const uint16_t*)w, amax_scratch, K, N, rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  quantize_cols_kernel<<<dim3((unsigned)((N + 63) / 64), (unsigned)((K + 63) / 64)), kThreads,
                         0, st>>>((const uint16_t*)w, amax_scratch, (uint8_t*)codes_nk, scales,
                                  K, N);
  return cudaGetLastError();
}

}  // namespace swg
