// Large-M path on the tensor cores (bf16): a persistent tcgen05 GEMM whose
// epilogue applies SwiGLU to the accumulator tile before one bf16 store.
//
// "Tile-Level Activation Overlap for Efficient LLM Inference" fuses SwiGLU
// into the GEMM at tile level so that neither Gate nor Up is ever written to
// HBM; its Kernel-2 interleaves the gate and up weight columns so one GEMM
// tile holds matching gate/up column pairs and its epilogue emits
// SiLU(gate) * up.  This kernel keeps that idea and re-does the rest for
// sm_103a:
//   * an output tile is 128 rows x 128 columns of h; its accumulator is
//     128 x 256 f32 in TMEM: columns 0-127 = x.W_gate, 128-255 = x.W_up for
//     the same 128 output columns (the interleave happens per 64-column TMA
//     box while loading; W_gate and W_up stay separate row-major arrays);
//   * A = x tile (K-major), B = the four weight boxes (MN-major, read straight
//     from the row-major weights), both TMA-staged in a 4-stage ring
//     (6 stages on a CTA pair);
//   * one thread issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM
//     accumulators, so the epilogue of tile i overlaps the MMAs of tile i+1
//     (the overlap the paper gets from ping-pong warp groups);
//   * the epilogue (4 warps, one accumulator row per thread) reads gate and up
//     columns with tcgen05.ld, computes silu(g) * u in f32, rounds to bf16 into
//     a 128-byte-swizzled staging tile and TMA-stores it.
// Tiles are visited band by band (a band = a few 128/256-row blocks),
// column-block-major inside a band, so the CTAs running at the same time
// share weight columns and x rows through L2 (tile_coords).
//
// Above 128 rows the kernel runs on CTA pairs (2-CTA clusters, tcgen05
// cta_group::2): a tile is 256 rows, each CTA loads its 128 rows of x and
// half of the weight boxes (gate in rank 0, up in rank 1), and one M = 256
// MMA stream fills both CTAs' TMEM.  Per CTA and k-block that is 32 KB of
// operands instead of 48 KB, so six stages fit and the L2 -> SM bytes per
// FLOP fall by a third (measured: prefill 480 vs 549 us per call).
//
// In its plain mode the same kernel computes the down projection
// y = h . W_down (+ residual) ("1 . Anatomie d'un transformeur sur GPU",
// section 1.6, kernels #10 and #11): the 256 accumulator columns are 256
// adjacent output columns, and the epilogue adds the residual and stores
// them in two 128-column passes.
#include <atomic>
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "tc_pair.cuh"

namespace swg {
namespace {

using namespace tc;

constexpr int kBM = 128;                        // output rows per CTA and tile
constexpr int kBN = 128;                        // output columns per tile
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kChunkBytes = 64 * kBK * 2;  // 8 KB: one 64-column weight box
constexpr uint32_t kStagingHalf = kBM * 128;    // 128 rows x 64 bf16
constexpr uint32_t kStagingBytes = 2 * kStagingHalf;
constexpr uint32_t kTmemCols = 512;             // two 128 x 256 f32 accumulators

// One CTA per tile (PAIR = false), or a 2-CTA cluster per 256-row tile whose
// MMAs run as cta_group::2 (PAIR = true).  A pair tile gives each CTA 128 rows
// of x and half of the 256 weight columns, so a CTA stages 32 KB per k-block
// instead of 48 KB: more stages fit, and the L2 -> SM bytes per FLOP drop by
// a third.
template <bool PAIR>
struct TileCfg {
  static constexpr int kBoxes = PAIR ? 2 : 4;   // 64-column weight boxes per CTA and k-block
  static constexpr uint32_t kBBytes = kBoxes * kChunkBytes;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
  static constexpr size_t kSmemBytes =
      1024 + (size_t)kStages * kStageBytes + kStagingBytes + 256;
};
static_assert(TileCfg<true>::kSmemBytes <= 232448, "pair tile exceeds shared memory");
static_assert(TileCfg<false>::kSmemBytes <= 232448, "tile exceeds shared memory");

struct TileArgs {
  int n_mb, n_kb, n_out;         // n_mb: row blocks of the tile height; n_out: output columns
  int n_nb, band;                // column blocks; row blocks per band (tile_coords)
  int M;
  const uint16_t* resid;         // plain mode: [M][n_out] added to the sums, or null
  int kmajor;                    // weights stored [n_out, K] instead of [K, n_out]
  int packed;                    // SwiGLU: one packed gate/up matrix (tm_wg = tm_wu)
  int seq;                       // SwiGLU, one CTA: gate then up, each an N = 128 k loop
  const float* sx;               // fp8: [M] row scales of x
  const float* sw_a;             // fp8: [n_out] column scales of W_gate
  const float* sw_b;             // fp8: [n_out] column scales of W_up
  unsigned* status;
  uint64_t timeout_ns;
  // Stream-K tail.  Tiles [0, dp_tiles) are done whole, round-robin over the
  // units (CTAs, or CTA pairs).  The k-blocks of the tiles after them form one
  // iteration space of sk_iters = (tiles - dp_tiles) * n_kb, cut into
  // contiguous ranges: sk_q + 1 iterations for each of the first sk_r units,
  // sk_q for the rest.
  int64_t dp_tiles, sk_iters, sk_q, sk_r;
  float* part;                   // partial tiles: slot (tile - dp_tiles + unit), rank, 8 x 8 x 128 x 4 f32
  unsigned* counters;            // arrivals per stream-K tile and rank; left at zero
};

constexpr int kPartFloats = kBM * 2 * kBN;   // one CTA's 128 x 256 f32 accumulator

// Row block mb and column block nb of tile t.  The row blocks are cut into
// bands of `band` (the last band may be shorter); tiles run band by band,
// column-block-major inside a band, so the tiles in flight at once share the
// x rows of one band and a few weight columns through L2.  With one band
// (band = n_mb) this is the plain column-block-major order.
__device__ __forceinline__ void tile_coords(const TileArgs& a, int64_t t, int& mb, int& nb) {
  const int64_t full = (int64_t)(a.n_mb / a.band) * a.band * a.n_nb;   // tiles in full bands
  if (t < full) {
    const int64_t per = (int64_t)a.band * a.n_nb;
    const int64_t b = t / per, l = t - b * per;
    nb = (int)(l / a.band);
    mb = (int)(b * a.band + (l - (int64_t)nb * a.band));
  } else {
    const int64_t rows = a.n_mb - (int64_t)(a.n_mb / a.band) * a.band;
    const int64_t l = t - full;
    nb = (int)(l / rows);
    mb = (int)((int64_t)(a.n_mb / a.band) * a.band + (l - (int64_t)nb * rows));
  }
}

// First stream-K iteration of unit u.
__device__ __forceinline__ int64_t sk_begin(const TileArgs& a, int64_t u) {
  return u * a.sk_q + (u < a.sk_r ? u : a.sk_r);
}

// Unit whose range holds stream-K iteration i.
__device__ __forceinline__ int64_t sk_unit_of(const TileArgs& a, int64_t i) {
  const int64_t big = a.sk_r * (a.sk_q + 1);
  return i < big ? i / (a.sk_q + 1) : a.sk_r + (i - big) / a.sk_q;
}

// The work items of one unit, in order: its whole tiles, then its stream-K
// range cut at tile boundaries.  An item is a tile and a k-block range.
struct WorkIter {
  int64_t t_dp, it, it_end;
  __device__ WorkIter(const TileArgs& a, int64_t unit) : t_dp(unit) {
    it = a.sk_iters ? sk_begin(a, unit) : 0;
    it_end = a.sk_iters ? sk_begin(a, unit + 1) : 0;
  }
  __device__ bool next(const TileArgs& a, int64_t n_units, int64_t& t, int& kb0, int& kb1) {
    if (t_dp < a.dp_tiles) {
      t = t_dp;
      kb0 = 0;
      kb1 = a.n_kb;
      t_dp += n_units;
      return true;
    }
    if (it < it_end) {
      const int64_t rel = it / a.n_kb;
      const int64_t stop = (rel + 1) * a.n_kb < it_end ? (rel + 1) * a.n_kb : it_end;
      t = a.dp_tiles + rel;
      kb0 = (int)(it - rel * a.n_kb);
      kb1 = (int)(stop - rel * a.n_kb);
      it = stop;
      return true;
    }
    return false;
  }
};

constexpr int kSwiGLU = 0;       // accumulator = 128 gate columns | 128 up columns
constexpr int kPlain = 1;        // accumulator = 256 adjacent output columns

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, unsigned* status,
                                           uint64_t timeout_ns) {
  int never = 0;
  return mbar_wait(bar, parity, &never, status, timeout_ns);
}

// FP8: e4m3 operands (kind::f8f6f4) and scaled sums.  A compile-time choice:
// one kernel issuing MMAs of two kinds behind a runtime branch measured
// 20-40 % slower on its bf16 work.
template <int MODE, bool PAIR, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
tile_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
               const __grid_constant__ CUtensorMap tm_wu, const __grid_constant__ CUtensorMap tm_h,
               const TileArgs a) {
  using C = TileCfg<PAIR>;
  constexpr int kStages = C::kStages;
  // output columns per tile, and where the 64-column B boxes come from
  constexpr int kOutCols = MODE == kSwiGLU ? kBN : 2 * kBN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint8_t* staging = stages + (size_t)kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kStagingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile unsigned* ticket_slot = reinterpret_cast<volatile unsigned*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // In a pair, rank 0 issues the MMAs for both CTAs; each CTA loads its own
  // 128 rows of x and its half of the weight columns and runs its own
  // epilogue on the 128 accumulator rows in its TMEM.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int64_t unit = PAIR ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
  const int64_t n_units = PAIR ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // rank 0's stage is full once its own bytes have landed and rank 1 has
      // relayed that its half has landed too
      mbar_init(&full[s], (PAIR && rank == 0) ? 2 : 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    // a pair's accumulator is free once both CTAs' epilogues have read it
    mbar_init(&tempty[0], PAIR ? 2 * kEpiThreads : kEpiThreads);
    mbar_init(&tempty[1], PAIR ? 2 * kEpiThreads : kEpiThreads);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
    tma_prefetch_desc(&tm_h);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();   // both CTAs' barriers and TMEM are ready
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The pair's MMAs address both TMEMs with one column address; if the two
  // allocations disagree, neither CTA does any work.
  bool skip = false;
  if constexpr (PAIR) {
    skip = ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), rank ^ 1u)) != tmem;
    if (skip && threadIdx.x == 0) atomicOr(a.status, kStatusPairTmem);
  }
  // The set-up above overlaps the previous kernel's tail; x and h are touched
  // only after it has finished.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer (each CTA) ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = !skip;
      WorkIter w(a, unit);
      int64_t t;
      int kb0, kb1;
      // Sequential order (seq): the tile's k loop runs twice, first with
      // only the two gate boxes per stage, then with only the two up boxes.
      const int n_ph = (MODE == kSwiGLU && !PAIR && !FP8 && a.seq) ? 2 : 1;
      const int n_box = n_ph == 2 ? 2 : C::kBoxes;
      const uint32_t stage_tx = kABytes + (uint32_t)n_box * kChunkBytes;
      while (ok && w.next(a, n_units, t, kb0, kb1)) {
        int mb, nb;
        tile_coords(a, t, mb, nb);
        const int row0 = mb * C::kTileRows + (int)rank * kBM;
        for (int ph = 0; ok && ph < n_ph; ++ph)
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)stage * C::kStageBytes;
          uint8_t* sb = st + kABytes;
          mbar_arrive_expect_tx(&full[stage], stage_tx);
          tma_load_2d(st, &tm_x, &full[stage], kb * kBK, row0);
#pragma unroll
          for (int q = 0; q < C::kBoxes; ++q) {
            // B boxes.  One CTA: SwiGLU -> gate 0-63, gate 64-127, up 0-63,
            // up 64-127 of the tile's columns; plain -> 4 x 64 adjacent
            // columns.  Pair: rank 0 holds accumulator columns 0-127 (gate,
            // or output columns 0-127), rank 1 columns 128-255 (up, or
            // output columns 128-255).  Sequential order: the two boxes of
            // this phase's matrix only.
            const bool up = PAIR ? rank == 1 : (n_ph == 2 ? ph == 1 : q >= 2);
            const CUtensorMap* m = (MODE == kSwiGLU && up) ? &tm_wu : &tm_wg;
            int col;
            if constexpr (PAIR)
              col = MODE == kSwiGLU ? nb * kBN + 64 * q : nb * kOutCols + (int)rank * kBN + 64 * q;
            else
              col = MODE == kSwiGLU ? nb * kBN + 64 * (q & 1) : nb * kOutCols + 64 * q;
            // packed gate/up matrix: gate block at 2 col, up block at 2 col + 64
            if (MODE == kSwiGLU && a.packed) col = 2 * col + (up ? 64 : 0);
            uint8_t* dst = sb + q * kChunkBytes;
            if (q < n_box) {
              if (a.kmajor)
                tma_load_2d(dst, m, &full[stage], kb * kBK, col);
              else
                tma_load_2d(dst, m, &full[stage], col, kb * kBK);
            }
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (issued > 0 && !ok) {
        // let the loads still in flight land before the CTA can exit
        const int64_t first = issued > kStages ? issued - kStages : 0;
        for (int64_t i = first; i < issued; ++i)
          wait_drain(&full[i % kStages], (uint32_t)((i / kStages) & 1), a.status, a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1 && (!PAIR || rank == 0)) {
    // ---------------- MMA issuer (the CTA, or rank 0 of the pair) ----------------
    if (lane == 0) {
      // A (x) is K-major; B (the weights) MN-major for [K, n_out] weights,
      // K-major for [n_out, K] weights.
      // (FP8: e4m3 codes, K-major; one MMA takes 32 of them, the same 32 bytes)
      constexpr int kMmaM = PAIR ? 2 * kBM : kBM;
      const uint32_t idesc = FP8        ? idesc_e4m3_f32(kMmaM, 2 * kBN)
                             : a.kmajor ? idesc_bf16_f32(kMmaM, 2 * kBN, false, false)
                                        : idesc_bf16_f32(kMmaM, 2 * kBN, false, true);
      const uint32_t b_step = a.kmajor ? 32u : 2048u;
      const uint32_t b_lbo = a.kmajor ? 16u : kChunkBytes;
      // sequential order: two N = 128 k loops per tile (gate into accumulator
      // columns 0-127, then up into 128-255)
      const int n_ph = (MODE == kSwiGLU && !PAIR && !FP8 && a.seq) ? 2 : 1;
      const uint32_t idesc_mma =
          n_ph == 2 ? idesc_bf16_f32(kMmaM, kBN, false, a.kmajor == 0) : idesc;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = !skip;
      WorkIter w(a, unit);
      int64_t t;
      int kb0, kb1;
      while (ok && w.next(a, n_units, t, kb0, kb1)) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ph = 0; ok && ph < n_ph; ++ph)
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t d_tmem = tmem + (uint32_t)(acc * 2 * kBN + ph * kBN);
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + (size_t)stage * C::kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32u, 16u, 1024u);
            const uint64_t bd = smem_desc_sw128(b_addr + kk * b_step, b_lbo, 1024u);
            const uint32_t accumulate = (kb != kb0 || kk != 0) ? 1u : 0u;
            if constexpr (PAIR && FP8)
              mma_e4m3_pair(d_tmem, ad, bd, idesc, accumulate);
            else if constexpr (PAIR)
              mma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
            else if constexpr (FP8)
              mma_e4m3(d_tmem, ad, bd, idesc, accumulate);
            else
              mma_bf16(d_tmem, ad, bd, idesc_mma, accumulate);
          }
          // the stage is free again in both CTAs once these MMAs are done
          if constexpr (PAIR)
            mma_commit_pair_mc(&empty[stage], (uint16_t)0x3);
          else
            mma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          mma_commit_pair_mc(&tfull[acc], (uint16_t)0x3);
        else
          mma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if constexpr (PAIR)
        mma_commit_pair(drain);
      else
        mma_commit(drain);
      wait_drain(drain, 0, a.status, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- rank 1 of a pair: relay ----------------
    // Tell rank 0 when this CTA's half of each stage has landed.
    if constexpr (PAIR) {
      if (lane == 0) {
        const uint32_t full0 = mapa_shared(smem_u32(full), 0u);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = !skip;
        WorkIter w(a, unit);
        int64_t t;
        int kb0, kb1;
        while (ok && w.next(a, n_units, t, kb0, kb1)) {
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, a.status, a.timeout_ns)) {
              ok = false;
              break;
            }
            mbar_arrive_remote(full0 + (uint32_t)stage * 8u);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 2..5 (each CTA) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // accumulator row = output row in this CTA's rows
    const int et = threadIdx.x - 64;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    constexpr int kPasses = MODE == kSwiGLU ? 1 : 2;   // 128 output columns per pass
    // rank 1 tells rank 0's MMA issuer that an accumulator has been read
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(tempty), 0u) : 0u;
    constexpr int kRanks = PAIR ? 2 : 1;
    int acc = 0;
    uint32_t acc_phase = 0;
    WorkIter w(a, unit);
    int64_t t;
    int kb0, kb1;
    while (!skip && w.next(a, n_units, t, kb0, kb1)) {
      int mb, nb;
      tile_coords(a, t, mb, nb);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, a.status, a.timeout_ns)) break;
      tc_fence_after();
      const int row_base = mb * C::kTileRows + (int)rank * kBM;
      const int64_t grow = (int64_t)row_base + row;       // output row of this thread
      const uint32_t acc_col = (uint32_t)(acc * 2 * kBN);
      // A stream-K item holds part of the tile's k range.  This CTA stores its
      // partial accumulator in its slot (slot = tile - dp_tiles + unit, so the
      // units of one tile have consecutive slots), frees the accumulator and
      // takes a ticket; the last of the tile's units to arrive adds all the
      // partials in k order and runs the epilogue on the sum.
      const bool whole = kb0 == 0 && kb1 == a.n_kb;
      const float* seg0 = nullptr;
      int nseg = 0;
      if (!whole) {
        const int64_t rel = t - a.dp_tiles;
        float* mine = a.part + ((rel + unit) * kRanks + rank) * (int64_t)kPartFloats;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_off + acc_col + (uint32_t)(c * 32), v);
          tmem_wait_ld();
          // slot layout [32-column chunk][4-column group][row][4]: a warp's
          // store covers 512 contiguous bytes
          float4* dst = reinterpret_cast<float4*>(mine + ((int64_t)c * 8 * kBM + row) * 4);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(dst + i * kBM, make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                        __uint_as_float(v[4 * i + 2]),
                                        __uint_as_float(v[4 * i + 3])));
        }
        tc_fence_before();
        if (PAIR && rank == 1)
          mbar_arrive_remote(tempty0 + (uint32_t)acc * 8u);
        else
          mbar_arrive(&tempty[acc]);
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (et == 0) *ticket_slot = atomicAdd(a.counters + rel * kRanks + rank, 1u);
        named_bar_sync(1, kEpiThreads);
        const unsigned ticket = *ticket_slot;
        const int64_t u_first = sk_unit_of(a, rel * a.n_kb);
        nseg = (int)(sk_unit_of(a, rel * a.n_kb + a.n_kb - 1) - u_first + 1);
        if (ticket + 1u != (unsigned)nseg) {
          // not the last (or a counter left over by a call that gave up)
          if (ticket >= (unsigned)nseg && et == 0) atomicOr(a.status, kStatusStaleCounter);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
          continue;
        }
        __threadfence();
        if (et == 0) a.counters[rel * kRanks + rank] = 0u;   // left at zero for the next call
        seg0 = a.part + ((rel + u_first) * kRanks + rank) * (int64_t)kPartFloats;
      }
      for (int pass = 0; pass < kPasses; ++pass) {
        if (et == 0) bulk_wait_read0();   // the previous store has read the staging tile
        __syncwarp();
        named_bar_sync(1, kEpiThreads);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t g[32], u[32];
          if (whole) {
            const uint32_t col0 = acc_col + (uint32_t)(pass * kBN + ch * 32);
            tmem_ld_x32(tmem + lane_off + col0, g);
            if constexpr (MODE == kSwiGLU) tmem_ld_x32(tmem + lane_off + col0 + kBN, u);
            tmem_wait_ld();
          } else {
            // sum of the tile's partials, in k order
            float gs[32], us[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) gs[i] = us[i] = 0.f;
            const int cg = pass * 4 + ch;   // 32-column chunk of the gate (or output) columns
#pragma unroll 1
            for (int sg = 0; sg < nseg; ++sg) {
              const float* sp = seg0 + (int64_t)sg * kRanks * kPartFloats;
              const float4* pg =
                  reinterpret_cast<const float4*>(sp + ((int64_t)cg * 8 * kBM + row) * 4);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 q = __ldcg(pg + i * kBM);
                gs[4 * i] += q.x; gs[4 * i + 1] += q.y; gs[4 * i + 2] += q.z; gs[4 * i + 3] += q.w;
              }
              if constexpr (MODE == kSwiGLU) {
                const float4* pu =
                    reinterpret_cast<const float4*>(sp + ((int64_t)(cg + 4) * 8 * kBM + row) * 4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 q = __ldcg(pu + i * kBM);
                  us[4 * i] += q.x; us[4 * i + 1] += q.y; us[4 * i + 2] += q.z; us[4 * i + 3] += q.w;
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __float_as_uint(gs[i]);
              u[i] = __float_as_uint(us[i]);
            }
          }
          if constexpr (FP8) {
            // FP8: the sums times sx[row] sw[column] (gate / output columns
            // from sw_a, up columns from sw_b)
            const float sxm = grow < a.M ? a.sx[grow] : 0.f;
            const int64_t c0 = (int64_t)nb * kOutCols + pass * kBN + ch * 32;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), su = sg;
              if (c0 + 4 * v < a.n_out) {   // n_out is a multiple of 8
                sg = reinterpret_cast<const float4*>(a.sw_a + c0)[v];
                if constexpr (MODE == kSwiGLU) su = reinterpret_cast<const float4*>(a.sw_b + c0)[v];
              }
              const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                g[4 * v + e] = __float_as_uint(__uint_as_float(g[4 * v + e]) * (sxm * sgv[e]));
                if constexpr (MODE == kSwiGLU)
                  u[4 * v + e] = __float_as_uint(__uint_as_float(u[4 * v + e]) * (sxm * suv[e]));
              }
            }
          }
          float rv[32];
          if constexpr (MODE == kPlain) {
            // residual row segment: 32 bf16 of this output row
            const int64_t c0 = (int64_t)nb * kOutCols + pass * kBN + ch * 32;
            const bool has = a.resid && grow < a.M && c0 < a.n_out;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w = make_uint4(0u, 0u, 0u, 0u);
              if (has && c0 + 8 * v < a.n_out)
                w = *reinterpret_cast<const uint4*>(a.resid + grow * a.n_out + c0 + 8 * v);
              rv[8 * v + 0] = bf16_lo(w.x); rv[8 * v + 1] = bf16_hi(w.x);
              rv[8 * v + 2] = bf16_lo(w.y); rv[8 * v + 3] = bf16_hi(w.y);
              rv[8 * v + 4] = bf16_lo(w.z); rv[8 * v + 5] = bf16_hi(w.z);
              rv[8 * v + 6] = bf16_lo(w.w); rv[8 * v + 7] = bf16_hi(w.w);
            }
          }
          uint8_t* rowp = staging + (ch >> 1) * kStagingHalf + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 8 * i + 2 * e;
              float o0, o1;
              if constexpr (MODE == kSwiGLU) {
                o0 = silu_fast(__uint_as_float(g[q])) * __uint_as_float(u[q]);
                o1 = silu_fast(__uint_as_float(g[q + 1])) * __uint_as_float(u[q + 1]);
              } else {
                o0 = __uint_as_float(g[q]) + rv[q];
                o1 = __uint_as_float(g[q + 1]) + rv[q + 1];
              }
              w[e] = pack_bf16x2(o0, o1);
            }
            const int chunk = ((ch & 1) * 4 + i) ^ (row & 7);   // 128-byte swizzle
            *reinterpret_cast<uint4*>(rowp + chunk * 16) = v;
          }
        }
        if (whole && pass == kPasses - 1) {
          // every accumulator column of this buffer has been read
          tc_fence_before();
          if (PAIR && rank == 1)
            mbar_arrive_remote(tempty0 + (uint32_t)acc * 8u);
          else
            mbar_arrive(&tempty[acc]);
        }
        fence_async_smem();
        __syncwarp();
        named_bar_sync(1, kEpiThreads);
        if (et == 0) {
          // (rank 1 of a pair whose 256-row tile sticks out past M may have
          // no rows to store)
          const int c0 = nb * kOutCols + pass * kBN;
          if (row_base < a.M) {
            if (c0 < a.n_out) tma_store_2d(&tm_h, staging, c0, row_base);
            if (c0 + 64 < a.n_out)
              tma_store_2d(&tm_h, staging + kStagingHalf, c0 + 64, row_base);
          }
          bulk_commit();
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (et == 0) bulk_wait0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA of a pair leaves (or frees its TMEM) while the other may still
  // signal its barriers or read its shared memory.
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}


}  // namespace

TilePlan plan_tile(int64_t M, int64_t K, int64_t n_out, int num_sms, bool plain,
                   int max_pairs, const Tuning& tn) {
  TilePlan p{};
  const int64_t cols = plain ? 2 * kBN : kBN;
  p.plain = plain;
  // 2-CTA tiles wherever there is more than one 128-row block;
  // SWIGLU_TILE_PAIR = 0 / 1 forces one mode.
  const int forced = tn.tile_pair;
  p.pair = forced >= 0 ? forced != 0 : M > kBM;
  if (num_sms < 2 || max_pairs < 1) p.pair = false;
  // The SwiGLU paper's Kernel-1 order (gate tile, then up tile, instead of
  // the interleaved gate|up accumulator): kept to compare the two, never
  // chosen by default (measured slower); SWIGLU_TILE_SEQ = 1 selects it, on
  // single-CTA tiles.
  p.seq = !plain && tn.tile_seq == 1;
  if (p.seq) p.pair = false;
  const int64_t rows = p.pair ? 2 * kBM : kBM;
  p.n_mb = (M + rows - 1) / rows;
  p.n_nb = (n_out + cols - 1) / cols;
  p.n_kb = (K + kBK - 1) / kBK;
  p.tiles = p.n_mb * p.n_nb;
  // units: CTAs, or CTA pairs, that run at once
  int64_t units = p.pair ? (num_sms / 2 < max_pairs ? num_sms / 2 : max_pairs) : num_sms;
  if (units < 1) units = 1;
  // Banded tile order.  The tiles in flight at once (one per unit) share the
  // x rows of one band, which every wave of the band reads again, while each
  // weight column block is used by one wave only.  So a band holds as many
  // row blocks as keep its x rows within a quarter of L2 (32 MB), evened
  // out over the bands.  Measured at d = 8192, d_ff = 29568, M = 8192 (32
  // row blocks of 4 MB; calls back to back): one band 5148 us (x re-read
  // from DRAM for every wave: 16.75 GB of DRAM reads per call against
  // 1.59 GB of algorithmic bytes), bands of 16 / 11 / 8 row blocks 4731 /
  // 4569 / 4413 us.  Prefill (d = 4096, 16 row blocks of 2 MB) and d = 8192,
  // M = 2048 keep one band, their fastest.  SWIGLU_TILE_BAND overrides.
  {
    const int64_t xr = rows * K * 2;   // bytes of x per row block
    const int64_t budget = (int64_t)32 << 20;
    int64_t band = xr > 0 ? budget / xr : p.n_mb;
    if (band < 1) band = 1;
    if (band > p.n_mb) band = p.n_mb;
    if (band > 0) {
      const int64_t nbands = (p.n_mb + band - 1) / band;
      band = (p.n_mb + nbands - 1) / nbands;
    }
    if (tn.tile_band > 0) band = tn.tile_band < p.n_mb ? tn.tile_band : p.n_mb;
    p.band = band > 0 ? band : 1;
  }
  p.dp_tiles = p.tiles;
  // Stream-K tail.  With W full waves and a partial one, the last wave plus
  // one full wave (all tiles if W = 0) are split along K over the units, in
  // equal contiguous shares of (tile, k-block) iterations; the rest are done
  // whole.  With W = 0 a tile is split over at most 4 units
  // (SWIGLU_TILE_SK_SPLIT), which bounds the partials its final reduction
  // reads.  Measured on GB300, it pays only where whole tiles would leave
  // most units idle: the down projection at d = 4096 with M = 64 / 256 (16
  // tiles) ran in 48 / 52 us instead of 97 / 84 us.  Where the tiles fill
  // >= 3/4 of a wave or more than one wave it was 4-35 % slower: units at
  // different k offsets no longer share weight and x tiles through L2, so
  // operands are re-read from DRAM.  So it is used when whole tiles keep
  // < 30 % of the units busy and each unit gets >= 4 k-blocks.
  // SWIGLU_TILE_SK = 0 / 1 forces it off / on (on: wherever there is a
  // partial wave).
  const int forced_sk = tn.tile_sk;
  int max_split = tn.tile_sk_split >= 0 ? tn.tile_sk_split : 4;
  if (max_split < 2) max_split = 2;
  const int64_t waves = p.tiles / units, rem = p.tiles % units;
  if (p.tiles > 0 && p.n_kb > 0 && rem != 0 && forced_sk != 0) {
    const int64_t sk_tiles = waves >= 1 ? units + rem : p.tiles;
    int64_t g = units;
    if (waves == 0 && p.tiles * max_split < g) g = p.tiles * max_split;
    const int64_t iters = sk_tiles * p.n_kb;
    const int64_t q = iters / g;
    const double busy = (double)p.tiles / (double)((waves + 1) * units);
    const bool want = forced_sk == 1 ? q >= 1 : (busy < 0.3 && q >= 4);
    if (want && g > 1) {
      units = g;
      p.dp_tiles = p.tiles - sk_tiles;
      p.sk_iters = iters;
      p.sk_q = q;
      p.sk_r = iters % g;
    }
  }
  int64_t gu = p.sk_iters ? units : (p.tiles < units ? p.tiles : units);
  if (gu < 1) gu = 1;
  p.grid = (int)(p.pair ? 2 * gu : gu);
  if (p.sk_iters) {
    const int64_t ranks = p.pair ? 2 : 1;
    const int64_t sk_tiles = p.tiles - p.dp_tiles;
    p.counters_bytes = ((size_t)(sk_tiles * ranks) * sizeof(unsigned) + 255) / 256 * 256;
    // one slot per (stream-K tile, unit) pair that shares a tile: at most
    // sk_tiles + units slots (slot = tile - dp_tiles + unit)
    p.part_bytes = (size_t)((sk_tiles + gu) * ranks) * kPartFloats * sizeof(float);
  }
  return p;
}

cudaError_t tile_max_pairs(int* pairs) {
  auto kern = tile_tc_kernel<kSwiGLU, true, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)TileCfg<true>::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TileCfg<true>::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(pairs, kern, &cfg);
}

namespace {

template <int MODE, bool PAIR, bool FP8>
cudaError_t launch_mode(const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mu,
                        const CUtensorMap& mh, const TileArgs& a, int grid, cudaStream_t st) {
  using C = TileCfg<PAIR>;
  auto kern = tile_tc_kernel<MODE, PAIR, FP8>;
  static std::atomic<int> configured[64];   // zero: not yet set on that device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(1, std::memory_order_release);
  }
  // The grid is the plan's: the stream-K shares assume exactly this many
  // units (the plan already caps pairs at what can run at once).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, mx, mg, mu, mh, a);
}

}  // namespace

cudaError_t launch_tile_tc(const void* x, const void* wa, const void* wb, void* out,
                           const void* resid, int64_t M, int64_t K, int64_t n_out,
                           int wlayout, const TilePlan& p, float* part, unsigned* counters,
                           bool counters_clean, unsigned* status, uint64_t timeout_ns,
                           cudaStream_t st, const Fp8Scales* fp8) {
  if (p.tiles == 0 || K == 0) return cudaSuccess;
  if (p.sk_iters && (!part || !counters)) return cudaErrorInvalidValue;
  if (fp8 && wlayout != kWeightsNK) return cudaErrorInvalidValue;
  CUtensorMap mx, mg, mu, mh;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&mx, x, M, K, kBK, kBM)) != cudaSuccess) return e;
  const bool w_kmajor = wlayout == kWeightsNK, packed = wlayout == kWeightsPacked;
  if (packed && p.plain) return cudaErrorInvalidValue;
  const int64_t wr = w_kmajor ? n_out : K;
  const int64_t wc = w_kmajor ? K : (packed ? packed_cols(n_out) : n_out);
  if ((e = make_tmap_bf16_2d(&mg, wa, wr, wc, 64, 64)) != cudaSuccess) return e;
  if (p.plain || packed) {
    mu = mg;
  } else if ((e = make_tmap_bf16_2d(&mu, wb, wr, wc, 64, 64)) != cudaSuccess) {
    return e;
  }
  if ((e = make_tmap_bf16_2d(&mh, out, M, n_out, 64, kBM)) != cudaSuccess) return e;
  TileArgs a;
  a.n_mb = (int)p.n_mb;
  a.n_nb = (int)p.n_nb;
  a.band = (int)p.band;
  a.n_kb = (int)((K + kBK - 1) / kBK);
  a.n_out = (int)n_out;
  a.M = (int)M;
  a.resid = (const uint16_t*)resid;
  a.kmajor = w_kmajor ? 1 : 0;
  a.packed = packed ? 1 : 0;
  a.seq = p.seq ? 1 : 0;
  a.sx = fp8 ? fp8->sx : nullptr;
  a.sw_a = fp8 ? fp8->sw_a : nullptr;
  a.sw_b = fp8 ? fp8->sw_b : nullptr;
  a.status = status;
  a.timeout_ns = timeout_ns;
  a.dp_tiles = p.dp_tiles;
  a.sk_iters = p.sk_iters;
  a.sk_q = p.sk_q;
  a.sk_r = p.sk_r;
  a.part = part;
  a.counters = counters;
  // Stream-K arrival counters must be zero on entry.
  if (p.sk_iters && !counters_clean &&
      (e = cudaMemsetAsync(counters, 0, p.counters_bytes, st)) != cudaSuccess)
    return e;
  if (fp8 && p.plain)
    return p.pair ? launch_mode<kPlain, true, true>(mx, mg, mu, mh, a, p.grid, st)
                  : launch_mode<kPlain, false, true>(mx, mg, mu, mh, a, p.grid, st);
  if (fp8)
    return p.pair ? launch_mode<kSwiGLU, true, true>(mx, mg, mu, mh, a, p.grid, st)
                  : launch_mode<kSwiGLU, false, true>(mx, mg, mu, mh, a, p.grid, st);
  if (p.pair)
    return p.plain ? launch_mode<kPlain, true, false>(mx, mg, mu, mh, a, p.grid, st)
                   : launch_mode<kSwiGLU, true, false>(mx, mg, mu, mh, a, p.grid, st);
  return p.plain ? launch_mode<kPlain, false, false>(mx, mg, mu, mh, a, p.grid, st)
                 : launch_mode<kSwiGLU, false, false>(mx, mg, mu, mh, a, p.grid, st);
}

}  // namespace swg
