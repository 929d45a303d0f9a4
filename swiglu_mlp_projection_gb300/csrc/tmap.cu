// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query so the library does not link
// libcuda directly).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace swg {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;

void init_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  g_init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                cudaEnableDefault, &q);
  if (g_init_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
    g_init_err = cudaErrorSymbolNotFound;
  if (g_init_err == cudaSuccess) g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}
}  // namespace

// 2-D bf16 row-major tensor [rows, cols] (cols contiguous) with a box of
// box_cols x box_rows elements and 128-byte swizzle; out-of-range elements
// read as zero.  box_cols * 2 must be <= 128.  `l2_promo_bytes` (0, 64, 128
// or 256) is the L2 fill granularity the copies may promote to.
namespace {
// Encoded maps are cached: a map is a pure function of these fields (the base
// address, extents, box and promotion), so a hit is always valid, also after
// the memory at `base` has been freed and reused.
struct TmapKey {
  const void* base;
  int64_t rows, cols;
  int box_cols, box_rows, promo;
  bool operator==(const TmapKey& o) const {
    return base == o.base && rows == o.rows && cols == o.cols && box_cols == o.box_cols &&
           box_rows == o.box_rows && promo == o.promo;
  }
};
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kCacheSlots = 256;
TmapEntry g_cache[kCacheSlots];
std::mutex g_cache_mu;

size_t slot_of(const TmapKey& k) {
  uint64_t h = (uint64_t)(uintptr_t)k.base * 0x9E3779B97F4A7C15ull;
  h ^= (uint64_t)k.rows * 0xC2B2AE3D27D4EB4Full + (uint64_t)k.cols;
  h ^= (uint64_t)(k.box_cols * 131 + k.box_rows * 7 + k.promo) * 0x165667B19E3779F9ull;
  return (size_t)((h >> 17) % kCacheSlots);
}
}  // namespace

cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                              int box_cols, int box_rows, int l2_promo_bytes) {
  const TmapKey key{base, rows, cols, box_cols, box_rows, l2_promo_bytes};
  const size_t slot = slot_of(key);
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    if (g_cache[slot].valid && g_cache[slot].key == key) {
      *map = g_cache[slot].map;
      return cudaSuccess;
    }
  }
  std::call_once(g_once, init_encode);
  if (!g_encode) return g_init_err != cudaSuccess ? g_init_err : cudaErrorSymbolNotFound;
  // A tensor map needs every extent >= 1; callers never ask for empty maps.
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  const CUtensorMapL2promotion promo =
      l2_promo_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
      : l2_promo_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
      : l2_promo_bytes >= 64 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                             : CU_TENSOR_MAP_L2_PROMOTION_NONE;
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, promo,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_cache[slot].key = key;
  g_cache[slot].map = *map;
  g_cache[slot].valid = true;
  return cudaSuccess;
}

}  // namespace swg
