// Step a0: pack W_gate and W_up into one matrix whose 64-column blocks
// alternate, gate then up.
//
// "Tile-Level Activation Overlap for Efficient LLM Inference", Kernel-2,
// interleaves the gate and up weight columns once, before the GEMM, so that
// one GEMM tile holds matching gate/up columns.  Here the unit is the
// 64-column block that one TMA box (or one SIMT lane group) reads: with
// P = ceil(d_ff / 64) * 64, packed row k is
//     Wg[k, 0:64] | Wu[k, 0:64] | Wg[k, 64:128] | Wu[k, 64:128] | ...
// (2P elements; columns past d_ff are zero).  The copy is a streaming kernel:
// one thread moves one 16-byte chunk, consecutive threads consecutive chunks
// of the packed row, so both the reads and the writes are coalesced.
#include "common.cuh"
#include "internal.h"

namespace swg {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
pack_kernel(const uint4* __restrict__ wg, const uint4* __restrict__ wu, uint4* __restrict__ out,
            int64_t d, int64_t row_chunks_in, int64_t row_chunks_out, int64_t block_chunks) {
  // block_chunks: 16-byte chunks per 64-column block (8 for bf16, 16 for f32)
  const int64_t total = d * row_chunks_out;
  for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < total;
       q += (int64_t)gridDim.x * kThreads) {
    const int64_t k = q / row_chunks_out, c = q - k * row_chunks_out;
    const int64_t b = c / block_chunks, i = c - b * block_chunks;
    const int64_t src = (b >> 1) * block_chunks + i;   // chunk of the source row
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (src < row_chunks_in) v = ((b & 1) ? wu : wg)[k * row_chunks_in + src];
    out[q] = v;
  }
}

}  // namespace

int64_t packed_cols(int64_t d_ff) { return 2 * 64 * ((d_ff + 63) / 64); }

cudaError_t launch_pack(const void* wg, const void* wu, void* out, int64_t d, int64_t d_ff,
                        int dtype, int num_sms, cudaStream_t st) {
  const int64_t es = dtype == 1 ? 2 : 4;
  const int64_t row_in = d_ff * es / 16, row_out = packed_cols(d_ff) * es / 16;
  const int64_t total = d * row_out;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  pack_kernel<<<(unsigned)blocks, kThreads, 0, st>>>((const uint4*)wg, (const uint4*)wu,
                                                      (uint4*)out, d, row_in, row_out,
                                                      64 * es / 16);
  return cudaGetLastError();
}

}  // namespace swg
