// Inline-PTX building blocks for tensor-core kernels that run on a CTA pair
// (tcgen05 cta_group::2), plus the cross-CTA mbarrier operations the pair
// uses to hand work between its two CTAs.
//
// The two CTAs of a 2-CTA cluster act as one MMA unit.
//   * An M = 256 MMA takes A rows 0-127 from cluster rank 0's shared memory
//     and rows 128-255 from rank 1's.
//   * It takes B columns 0..N/2-1 from rank 0 and N/2..N-1 from rank 1, at the
//     same shared-memory offsets in both CTAs.
//   * It writes accumulator rows 0-127 to rank 0's TMEM and rows 128-255 to
//     rank 1's.
// One warp of each CTA allocates and frees the TMEM together; one thread of
// rank 0 issues the MMAs.  A kernel uses either these forms or the cta_group::1
// forms of tc_common.cuh, never both.
#pragma once

#include "tc_common.cuh"

namespace swg {

// Bit of the device error word (beside kStatusTimeout and kStatusStaleCounter):
// the two CTAs of a pair got different TMEM addresses, so the pair computed
// nothing.
enum : unsigned { kStatusPairTmem = 4u };

namespace tc {

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Arrive on an mbarrier of another CTA of the cluster (address from
// mapa_shared), with the default release semantics at CTA scope, as the
// waiting side uses.  (The .release.cluster form measured 2.3x slower
// end to end in the pair tile kernel, where it sits on the per-stage path.)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

// D[tmem of both CTAs] (+)= A x B over the pair; issued by one thread of rank 0.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same on e4m3 operands (kind::f8f6f4, idesc_e4m3_f32).
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// When all pair MMAs this thread issued before it complete, arrive once on the
// mbarrier at `bar`'s offset in every CTA of `cta_mask` (bit i = cluster rank i).
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

}  // namespace tc
}  // namespace swg
