// Self-test of the bounded device-side waits used by the tensor-core kernels.
#include "swiglu.h"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {
namespace {

// One CTA waits, through the same bounded wait the kernels use, on an
// mbarrier that nothing ever arrives on.  The wait gives up after
// `timeout_ns`, sets the device error word and the kernel returns normally.
__global__ void wait_timeout_kernel(unsigned* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);
  __syncthreads();
}

}  // namespace
}  // namespace swg

using namespace swg;

extern "C" int swiglu_selftest_wait_timeout(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000)
    return api_fail(SWIGLU_ERR_INVALID_ARG, "timeout_ms must be in 1..10000");
  int dev = 0, num_sms = 0;
  int v = api_current_device(&dev, &num_sms);
  if (v != SWIGLU_OK) return v;
  unsigned* status = api_status_word(dev);
  if (!status) return api_fail(SWIGLU_ERR_CUDA, "device status word unavailable");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = (cudaStream_t)stream;
  cudaError_t e = cudaLaunchKernelEx(&cfg, wait_timeout_kernel, status,
                                     (uint64_t)timeout_ms * 1000000ull);
  if (e != cudaSuccess) return api_cuda_fail(e, "kernel launch");
  api_clear_error();
  return SWIGLU_OK;
}
