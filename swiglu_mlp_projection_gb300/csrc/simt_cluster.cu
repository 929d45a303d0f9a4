// Cluster form of the SIMT path, for the smallest calls: one row of x on
// small weights (at most 32 MB, d <= 2048, e.g. the f32 decode step at
// d = 512), where a call moves a few MB and its time is set by latency, not
// by bandwidth.
//
// It computes the same sums as the split-K kernel of "Ou part le temps d'un
// token" (section "Un kernel pour les matrices etroites": the grid is cut
// along the weights, and the K slices of a column block are added in a fixed
// order), and applies SiLU * up only once they are complete, as that page's
// slice-reduction pass does.  What changes is where the slices meet:
//   * the S K slices of a column block (S = 8, or 7 ... 4 where the S = 8
//     clusters would not all fit at once) are one thread-block cluster; each
//     CTA stores its partial sums into the shared memory of the cluster's
//     rank 0 (distributed shared memory), and after one cluster barrier rank
//     0 adds the S partials in rank (= k) order and applies the epilogue;
//     the other CTAs exit at the barrier, since nobody reads their shared
//     memory.  No workspace, no arrival counter, no second pass through L2 -- the
//     page's "Ce qui reste : les lancements" finds such fixed costs to be
//     most of a small product's time;
//   * a column block is 128 bytes wide (32 f32 or 64 bf16 columns), so the
//     grid holds 4-8 CTAs per SM, and every thread issues all of its weight
//     loads (at most 8 rows of both matrices, 16 bytes each) and the x values
//     of those rows before it uses any: the whole call is in flight at once.  Eight lanes cover one 128-byte
//     row segment, so each warp load reads four full 128-byte lines.
// Sums per thread in k order, then across the four row groups of a warp
// (a fixed shuffle tree), across the 8 warps in warp order and across the
// cluster in rank order: the result is the same bits on every run.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace swg {

namespace {

constexpr int kThreads = 256;
constexpr int kLanesPerRow = 8;                       // 8 x 16 B = one 128-byte row segment
constexpr int kGroups = kThreads / kLanesPerRow;      // 32 rows of W in flight per pass
constexpr int kMaxRows = 8;                           // k rows per thread and matrix, at most
constexpr int kMaxK = kGroups * kMaxRows;             // 256 k per CTA at most (d <= 2048)
constexpr int kMaxS = 8;                              // CTAs per cluster (K slices), at most
constexpr int kMinS = 4;
constexpr int64_t kMaxWeightBytes = (int64_t)32 << 20;

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

// grid.x = column blocks x KS (a cluster = the KS K slices of one column
// block), grid.y = chunks of RC rows of x.  ROWS: k rows of W per thread
// (kn <= 32 ROWS), all in flight at once.  One row of x keeps 4 CTAs (1024
// threads) resident per SM, so that a call of 4 CTAs per SM runs in one wave.
template <bool BF16, int RC, int ROWS, int KS>
__global__ void __launch_bounds__(kThreads, (RC == 1 && ROWS <= 4) ? 4 : 2)
simt_cluster_kernel(const void* __restrict__ x_, const void* __restrict__ wg_,
                    const void* __restrict__ wu_, void* __restrict__ h_, int M, int d,
                    int d_ff, int packed) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int C = kLanesPerRow * VEC;   // columns of a block
  constexpr int ES = BF16 ? 2 : 4;
  __shared__ float red[kThreads / 32][RC][2][C];
  // rank 0 only: every slice's sums, written by their CTAs through
  // distributed shared memory
  __shared__ __align__(16) float part[KS][RC][2][C];

  const int rank = (int)tc::cluster_ctarank();        // = blockIdx.x % KS
  const int cb = blockIdx.x / KS;
  const int row0 = blockIdx.y * RC;
  const int k0 = (int)((int64_t)rank * d / KS), k1 = (int)((int64_t)(rank + 1) * d / KS);
  const int l8 = threadIdx.x & 7, grp = threadIdx.x >> 3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = cb * C + l8 * VEC;
  const bool valid = col < d_ff;

  // Before the dependency wait, one lane per 128-byte row segment prefetches
  // this thread group's weight rows into L2: a prefetch only reads, and L2 is
  // where every write lands, so it is safe while the previous kernel runs,
  // and the weight stream starts during that kernel's tail (measured, CUDA-
  // graph replay with 2 GiB of weights rotating: bf16 d = 896 at M = 1 in
  // 4.81 us against 5.28 us, the f32 decode step d = 512 in 3.19 against
  // 3.65 us).
  if (valid && l8 == 0) {
    const int gcol = packed ? col + (col & ~63) : col;
    const int ucol = packed ? gcol + 64 : col;
    const char* wg = (const char*)wg_ + (size_t)gcol * ES;
    const char* wu = (const char*)wu_ + (size_t)ucol * ES;
    const size_t row_bytes = (size_t)(packed ? 128 * ((d_ff + 63) / 64) : d_ff) * ES;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int kk = k0 + grp + kGroups * i;
      if (kk < k1) {
        tc::prefetch_l2(wg + (size_t)kk * row_bytes);
        tc::prefetch_l2(wu + (size_t)kk * row_bytes);
      }
    }
  }
  // Launched with programmatic stream serialisation: x and h may belong to
  // the previous kernel until this wait.
  tc::pdl_wait();
  tc::pdl_launch_dependents();

  // All loads first: rows k0 + grp + 32 i of both matrices, and the x values
  // of those rows (rows of x past M read as 0).
  uint4 vg[ROWS], vu[ROWS];
  float xv[ROWS][RC];
  if (valid) {
    // packed weights: gate block b of 64 columns at packed column 128 b, up
    // at 128 b + 64 (a block of 32 or 64 columns never straddles two)
    const int gcol = packed ? col + (col & ~63) : col;
    const int ucol = packed ? gcol + 64 : col;
    const char* wg = (const char*)wg_ + (size_t)gcol * ES;
    const char* wu = (const char*)wu_ + (size_t)ucol * ES;
    const size_t row_bytes = (size_t)(packed ? 128 * ((d_ff + 63) / 64) : d_ff) * ES;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int kk = k0 + grp + kGroups * i;
      if (kk < k1) {
        vg[i] = ldg_stream_v4(wg + (size_t)kk * row_bytes);
        vu[i] = ldg_stream_v4(wu + (size_t)kk * row_bytes);
      }
    }
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int kk = k0 + grp + kGroups * i;
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        float v = 0.f;
        if (kk < k1 && row0 + r < M) {
          const size_t idx = (size_t)(row0 + r) * d + kk;
          if constexpr (BF16)
            v = bf16_lo(__ldg((const unsigned short*)x_ + idx));
          else
            v = __ldg((const float*)x_ + idx);
        }
        xv[i][r] = v;
      }
    }
  }

  float accg[RC][VEC], accu[RC][VEC];
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int v = 0; v < VEC; ++v) accg[r][v] = accu[r][v] = 0.f;
  if (valid) {
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int kk = k0 + grp + kGroups * i;
      if (kk < k1) {
        float fg[VEC], fu[VEC];
        unpack16<BF16>(vg[i], fg);
        unpack16<BF16>(vu[i], fu);
#pragma unroll
        for (int r = 0; r < RC; ++r) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            accg[r][v] = fmaf(xv[i][r], fg[v], accg[r][v]);
            accu[r][v] = fmaf(xv[i][r], fu[v], accu[r][v]);
          }
        }
      }
    }
  }
  // The four row groups of a warp hold the same columns: lanes l, l^8, l^16,
  // l^24.  A fixed two-step tree leaves the same sum in all four.
#pragma unroll
  for (int r = 0; r < RC; ++r)
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      accg[r][v] += __shfl_xor_sync(0xffffffffu, accg[r][v], 8);
      accu[r][v] += __shfl_xor_sync(0xffffffffu, accu[r][v], 8);
      accg[r][v] += __shfl_xor_sync(0xffffffffu, accg[r][v], 16);
      accu[r][v] += __shfl_xor_sync(0xffffffffu, accu[r][v], 16);
    }
  if (lane < kLanesPerRow) {
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        red[warp][r][0][l8 * VEC + v] = accg[r][v];
        red[warp][r][1][l8 * VEC + v] = accu[r][v];
      }
  }
  __syncthreads();
  // this slice's sums over the 8 warps, in warp order, stored into rank 0's
  // shared memory (slot `rank`)
  const uint32_t part0 = tc::mapa_shared(tc::smem_u32(&part[rank][0][0][0]), 0u);
  for (int t = threadIdx.x; t < RC * 2 * C; t += kThreads) {
    const int c = t % C, gu = (t / C) & 1, r = t / (2 * C);
    float s = red[0][r][gu][c];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) s += red[w][r][gu][c];
    tc::st_shared_cluster_f32(part0 + (uint32_t)(((r * 2 + gu) * C + c) * 4), s);
  }
  tc::cluster_sync_all();   // every slice's sums are in rank 0's shared memory
  if (rank != 0) return;    // nobody reads the other CTAs' shared memory

  // Rank 0 adds the KS slices in rank (= k) order and applies the epilogue.
  constexpr int kChunks = RC * C / 4;
  for (int q = threadIdx.x; q < kChunks; q += kThreads) {
    const int r = q / (C / 4), c = (q - r * (C / 4)) * 4;
    const int row = row0 + r, j = cb * C + c;
    if (row >= M || j >= d_ff) continue;   // d_ff is a multiple of 4: chunks are whole
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const float4 a = *reinterpret_cast<const float4*>(&part[s][r][0][c]);
      const float4 b = *reinterpret_cast<const float4*>(&part[s][r][1][c]);
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
    }
    if constexpr (BF16) {
      uint2 o;
      o.x = pack_bf16x2(silu_fast(g.x) * u.x, silu_fast(g.y) * u.y);
      o.y = pack_bf16x2(silu_fast(g.z) * u.z, silu_fast(g.w) * u.w);
      *reinterpret_cast<uint2*>((uint16_t*)h_ + (size_t)row * d_ff + j) = o;
    } else {
      *reinterpret_cast<float4*>((float*)h_ + (size_t)row * d_ff + j) =
          make_float4(silu_accurate(g.x) * u.x, silu_accurate(g.y) * u.y,
                      silu_accurate(g.z) * u.z, silu_accurate(g.w) * u.w);
    }
  }
}

template <bool BF16, int RC, int ROWS, int KS>
cudaLaunchConfig_t launch_config(int64_t M, int64_t d_ff, cudaLaunchAttribute* attr,
                                 cudaStream_t st) {
  constexpr int C = kLanesPerRow * (BF16 ? 8 : 4);
  const int64_t n_cb = (d_ff + C - 1) / C;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = KS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_cb * KS), (unsigned)((M + RC - 1) / RC));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <bool BF16, int RC, int ROWS, int KS>
cudaError_t launch_rows(const void* x, const void* wg, const void* wu, void* h, int64_t M,
                        int64_t d, int64_t d_ff, bool packed, cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = launch_config<BF16, RC, ROWS, KS>(M, d_ff, attr, st);
  return cudaLaunchKernelEx(&cfg, simt_cluster_kernel<BF16, RC, ROWS, KS>, x, wg, wu, h, (int)M,
                            (int)d, (int)d_ff, packed ? 1 : 0);
}

// ROWS from the largest slice's k.  Clusters of fewer than 8 slices are
// planned only where a slice holds at most 4 rows per thread (slice_fits).
template <bool BF16, int RC, int KS>
cudaError_t launch_ks(const void* x, const void* wg, const void* wu, void* h, int64_t M,
                      int64_t d, int64_t d_ff, bool packed, cudaStream_t st) {
  const int64_t kn = (d + KS - 1) / KS;
  if (kn <= 2 * kGroups) return launch_rows<BF16, RC, 2, KS>(x, wg, wu, h, M, d, d_ff, packed, st);
  if (kn <= 4 * kGroups) return launch_rows<BF16, RC, 4, KS>(x, wg, wu, h, M, d, d_ff, packed, st);
  if constexpr (KS == kMaxS)
    return launch_rows<BF16, RC, 8, KS>(x, wg, wu, h, M, d, d_ff, packed, st);
  return cudaErrorInvalidValue;
}

template <bool BF16, int RC>
cudaError_t launch_rc(const void* x, const void* wg, const void* wu, void* h, int64_t M,
                      int64_t d, int64_t d_ff, int ks, bool packed, cudaStream_t st) {
  switch (ks) {
    case 8: return launch_ks<BF16, RC, 8>(x, wg, wu, h, M, d, d_ff, packed, st);
    case 7: return launch_ks<BF16, RC, 7>(x, wg, wu, h, M, d, d_ff, packed, st);
    case 6: return launch_ks<BF16, RC, 6>(x, wg, wu, h, M, d, d_ff, packed, st);
    case 5: return launch_ks<BF16, RC, 5>(x, wg, wu, h, M, d, d_ff, packed, st);
    case 4: return launch_ks<BF16, RC, 4>(x, wg, wu, h, M, d, d_ff, packed, st);
    default: return cudaErrorInvalidValue;
  }
}

// Can a cluster of ks slices serve a d-deep sum?  8 slices take up to 8 rows
// of W per thread (kMaxK = 256 k per slice); fewer slices only up to 4 rows,
// so that 4 CTAs still fit per SM.
bool slice_fits(int64_t d, int ks) {
  if (ks < kMinS || ks > kMaxS || d < ks) return false;
  const int64_t kn = (d + ks - 1) / ks;
  return ks == kMaxS ? kn <= kMaxK : kn <= 4 * kGroups;
}

template <int KS>
cudaError_t cap_of(int* n) {
  cudaLaunchAttribute attr[2];
  // one cluster's grid: the occupancy query asks how many such clusters fit
  cudaLaunchConfig_t cfg = launch_config<true, 1, 4, KS>(1, (int64_t)kLanesPerRow * 8, attr, 0);
  return cudaOccupancyMaxActiveClusters(n, simt_cluster_kernel<true, 1, 4, KS>, &cfg);
}

}  // namespace

int simt_cluster_plan(int64_t M, int64_t d, int64_t d_ff, int dtype, const Tuning& tn,
                      const int* caps) {
  if (tn.simt_cluster == 0) return 0;
  const int64_t e = dtype == 1 ? 2 : 4;
  const int C = kLanesPerRow * (dtype == 1 ? 8 : 4);
  // One row only (measured, graph replay): the f32 decode step d = 512,
  // d_ff = 2048 takes 4.6 us against 7.1 us on the split-K kernel.  Two or
  // four rows double or quadruple the accumulators, which halves the CTAs an
  // SM holds, and the call then needs two waves (bf16 d = 896: 12.4 / 15.4
  // us at M = 2 / 4 against 8.1 at M = 1).
  if (M != 1 || d_ff <= 0 || 2 * d * d_ff * e > kMaxWeightBytes) return 0;
  const int64_t n_cb = (d_ff + C - 1) / C;
  if (n_cb * kMaxS > (int64_t)INT32_MAX) return 0;
  if (tn.simt_cluster >= kMinS && tn.simt_cluster <= kMaxS)
    return slice_fits(d, tn.simt_cluster) ? tn.simt_cluster : 0;
  // The largest cluster whose n_cb clusters all run at once, 4 CTAs per SM
  // (caps[S]: clusters of S CTAs that fit).  A cluster of 8 must find 8 free
  // CTA slots in one GPC, and 4 per SM do not pack into whole 8-CTA clusters
  // on every GPC: e.g. the d = 896 model's 76 column blocks.
  if (caps)
    for (int ks = kMaxS; ks >= kMinS; --ks)
      if (slice_fits(d, ks) && (d + ks - 1) / ks <= 4 * kGroups && n_cb <= caps[ks]) return ks;
  return slice_fits(d, kMaxS) ? kMaxS : 0;
}

cudaError_t simt_cluster_caps(int caps[kSimtCapSlots]) {
  for (int i = 0; i < kSimtCapSlots; ++i) caps[i] = 0;
  cudaError_t e;
  if ((e = cap_of<8>(&caps[8])) != cudaSuccess) return e;
  if ((e = cap_of<7>(&caps[7])) != cudaSuccess) return e;
  if ((e = cap_of<6>(&caps[6])) != cudaSuccess) return e;
  if ((e = cap_of<5>(&caps[5])) != cudaSuccess) return e;
  return cap_of<4>(&caps[4]);
}

cudaError_t launch_simt_cluster(const void* x, const void* wg, const void* wu, void* h,
                                int64_t M, int64_t d, int64_t d_ff, int dtype, int ks,
                                bool packed, cudaStream_t st) {
  if (M == 0 || d_ff == 0) return cudaSuccess;
  if (M != 1) return cudaErrorInvalidValue;   // simt_cluster_plan serves one row
  if (!slice_fits(d, ks)) return cudaErrorInvalidValue;
  return dtype == 1 ? launch_rc<true, 1>(x, wg, wu, h, M, d, d_ff, ks, packed, st)
                    : launch_rc<false, 1>(x, wg, wu, h, M, d, d_ff, ks, packed, st);
}

}  // namespace swg
