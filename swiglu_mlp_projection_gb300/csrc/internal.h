// Internal interfaces between the C-ABI layer and the kernel launchers.
#pragma once

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
};

SimtPlan plan_simt(int64_t M, int64_t d, int64_t d_ff, int dtype, int num_sms);

// S1 (SIMT): partial sums of x.Wg and x.Wu per K slice.
cudaError_t launch_simt_partial(const void* x, const void* wg, const void* wu,
                                float* part, int64_t M, int64_t d, int64_t d_ff,
                                int dtype, const SimtPlan& p, cudaStream_t st);

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
constexpr int64_t kSimtMaxGridYZ = 65535;

}  // namespace swg
