// swiglu_up_noalloc: the SIMT split-K path with its partial sums in a fixed,
// library-held device array, for callers that cannot allocate device memory
// while the operation runs (see include/swiglu.h for who they are).  The
// kernels are the regular ones (skinny_simt.cu, reduce_swiglu.cu); only the
// origin of the scratch differs.
#include <cuda_runtime.h>

#include <mutex>
#include <stdio.h>

#include "swiglu.h"
#include "internal.h"

// The scratch array.  Every GPU that loads this library holds it until the
// process exits.  In host code this name is only a host-side stand-in, never
// a device address: kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SWIGLU_NOALLOC_SCRATCH_BYTES];

namespace swg {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on `dev` (the current device), looked
// up once per device.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return api_fail(SWIGLU_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return api_cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    if (!p) return api_fail(SWIGLU_ERR_CUDA, "cudaGetSymbolAddress(scratch) returned null");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SWIGLU_OK;
}

}  // namespace
}  // namespace swg

using namespace swg;

extern "C" int swiglu_up_noalloc(const void* x, const void* w_gate, const void* w_up, void* h,
                                 int64_t M, int64_t d, int64_t d_ff, int dtype, void* stream) {
  int v = api_validate(x, w_gate, w_up, h, M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  int dev = 0, num_sms = 0;
  if ((v = api_current_device(&dev, &num_sms)) != SWIGLU_OK) return v;
  if (M == 0 || d_ff == 0) {
    api_clear_error();
    return SWIGLU_OK;
  }
  const SimtPlan p = plan_simt(M, d, d_ff, dtype, num_sms);
  if (p.slices > kSimtMaxGridYZ || p.row_chunks > kSimtMaxGridYZ)
    return api_fail(SWIGLU_ERR_UNSUPPORTED, "shape exceeds the grid limits of the SIMT path");
  const size_t need = partial_elems(p.slices, M, d_ff) * sizeof(float);
  if (need > SWIGLU_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof msg, "needs %zu bytes of scratch; the fixed scratch holds %zu",
             need, (size_t)SWIGLU_NOALLOC_SCRATCH_BYTES);
    return api_fail(SWIGLU_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  if ((v = scratch_address(dev, &scratch)) != SWIGLU_OK) return v;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_simt_partial(x, w_gate, w_up, (float*)scratch, M, d, d_ff, dtype, p, st);
  if (e == cudaSuccess)
    e = launch_reduce_swiglu((const float*)scratch, h, M, d_ff, p.slices, dtype, num_sms, st);
  if (e != cudaSuccess) return api_cuda_fail(e, "kernel launch");
  api_clear_error();
  return SWIGLU_OK;
}
