// Device-side helpers shared by the kernels of the SwiGLU up-projection.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace swg {

// Bits of the device error word (see swiglu_check_device_status).
//   kStatusTimeout: a bounded wait gave up.
//   kStatusStaleCounter: an arrival counter did not start at zero (left over
//   by a call that gave up), so a column group was not reduced.
enum : unsigned { kStatusTimeout = 1u, kStatusStaleCounter = 2u };

// bf16 -> f32 is exact: a bf16 value is the upper half of a binary32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// f32 -> bf16, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// SiLU(z) = z * sigma(z) = z / (1 + e^-z) (Swish with beta = 1).  For
// z -> -inf, e^-z overflows to +inf and the quotient is -0, never NaN.
// The f32 path uses the accurate expf; the bf16 paths the fast __expf, whose
// error is far below half a bf16 ulp.
__device__ __forceinline__ float silu_accurate(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 16-byte streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace swg
