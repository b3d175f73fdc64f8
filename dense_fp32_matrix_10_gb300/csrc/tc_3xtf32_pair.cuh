// tc_3xtf32_pair.cuh -- the split-ahead 3xTF32 product on CTA pairs
// (tcgen05 .cta_group::2): one 256 x 128 (or 256 x 256) output tile per pair
// of CTAs.
//
// Same arithmetic as tc3_gemm_kernel's split-ahead form (TcConfig<1,1,1>):
// per k8 the three kind::tf32 MMAs a_small*b_big, a_big*b_small, a_big*b_big,
// accumulated in FP32 in tensor memory, promoted every 256 k into
// round-to-nearest FP32 registers.  What changes is who holds what:
//   * the pair's MMA is M = 256: the even CTA's shared memory holds A rows
//     0..127 of the tile, the odd CTA's rows 128..255, and each CTA's tensor
//     memory receives its own 128 rows of the accumulator;
//   * op(B)'s n-columns are split too: the first half in the even CTA, the
//     second in the odd one, and the tensor cores of both SMs read both.
// So at 256 x 128 each SM's stage is 48 KiB (its A rows, big and small, and
// its half of B, big and small) instead of 64 KiB, four stages fit instead
// of three, and each SM reads 6 KiB of operands per 128 x 128 x 8 of work
// instead of 8 KiB -- shared-memory operand reads bound the one-CTA kernel.
//
// Roles (per CTA, both CTAs of the pair):
//   warp 0       TMA producer of this CTA's slices; completion is counted on
//                the even CTA's `full` barrier (the even CTA's producer arms
//                it with the bytes of both CTAs);
//   warp 1       allocates 2 x BN TMEM columns (two accumulators; both CTAs,
//                same address); in the even CTA one thread issues the pair
//                MMAs and commits to the `empty` barriers of both CTAs and to
//                both CTAs' `acc_full`;
//   warps 4..    epilogue of this CTA's 128 rows, one warpgroup per 128
//                columns; they release an accumulator on the even CTA's
//                `acc_empty` (one arrival per epilogue warp of the pair);
//                with a folded operand they also compute its small parts;
//   warps 2, 3   idle, or converters with a folded operand at BN = 128.
// Every wait is bounded; a CTA leaves only after its peer has also finished
// (cluster barrier), so no copy or arrival lands in a CTA that has ended.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"
#include "tc_3xtf32.cuh"  // TcParams, tc_store_row, tile_coords

namespace sg {

// BN = 128: 256 x 128 pair tiles, 48 KiB stages, four of them.  BN = 256:
// 256 x 256 pair tiles (one 256 x 256 x 8 MMA per product term, each SM
// reading 8 KiB of operands per 128 x 256 x 8 of work), 64 KiB stages,
// three of them; the two 128-column halves of a CTA's rows go to two
// epilogue warpgroups.
// FOLD_A / FOLD_B: that operand is k-contiguous in memory, so its TMA tile
// is its own big part; instead of loading small parts written by a split pass,
// the CTA computes them in place (split_pair, the pass's arithmetic) once the
// big part has landed on the CTA's raw_full barrier, and then arrives on the
// pair's `full` barrier.  No split pass, no scratch for that operand, the
// same values.  The converters are the epilogue warps (idle between
// accumulator hand-overs; tcp_epilogue_fold interleaves both jobs) and, at
// BN = 128, warps 2 and 3 as well; every converter thread keeps its whole
// share of a stage in flight at once.
template <int BN_, bool FOLD_A_ = false, bool FOLD_B_ = false>
struct TcPairConfig {
  static constexpr bool FOLD_A = FOLD_A_, FOLD_B = FOLD_B_, FOLD = FOLD_A_ || FOLD_B_;
  static constexpr int BM = 256, BN = BN_, BK = 32;   // the pair's tile
  static_assert(BN == 128 || BN == 256, "pair tiles are 128 or 256 wide");
  static constexpr int B_ROWS = BN / 2;               // this CTA's n-rows of op(B)
  static constexpr int A_BYTES = 128 * 32 * 4;        // this CTA's A rows, one part
  static constexpr int B_BYTES = B_ROWS * 32 * 4;     // this CTA's half of B, one part
  static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
  static constexpr int A_BIG = 0, A_SMALL = A_BYTES, B_BIG = 2 * A_BYTES, B_SMALL = B_BIG + B_BYTES;
  static constexpr int STAGES = BN == 128 ? 4 : 3;
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
  // full[s] (used in the even CTA), empty[s], acc_full[2], acc_empty[2] (used
  // in the even CTA), drain, then raw_full[s] when a part is folded
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + (FOLD ? STAGES : 0);
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
  // warpgroup 0: producer, MMA, two idle warps; then one epilogue warpgroup
  // per 128 columns.  BN = 256 splits the registers with setmaxnreg.
  static constexpr int EPILOGUE_GROUPS = BN / 128;
  static constexpr int THREADS = 128 * (1 + EPILOGUE_GROUPS);
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr uint32_t IDESC = idesc_tf32(256, BN);
  static constexpr uint32_t IDESC_HALF = idesc_tf32(256, BN / 2);   // half-width units
  static constexpr int EPILOGUE_WARPS = 4 * EPILOGUE_GROUPS;
  static constexpr int CHUNK_KTILES = 8;   // k-slices (256 k) per promotion
  // converters: the epilogue warps, then (BN = 128, where warpgroup 0 keeps
  // its registers) warps 2 and 3
  static constexpr int CONV_SIDE_WARPS = (FOLD && BN_ == 128) ? 2 : 0;
  static constexpr int CONV_WARPS = FOLD ? EPILOGUE_WARPS + CONV_SIDE_WARPS : 0;
  static constexpr int CONV_THREADS = 32 * CONV_WARPS;
  // float4s per stage to convert, and per converter thread
  static constexpr int CONV_A_VEC = FOLD_A ? A_BYTES / 16 : 0;
  static constexpr int CONV_VEC = CONV_A_VEC + (FOLD_B ? B_BYTES / 16 : 0);
  static constexpr int CONV_PER_THREAD = FOLD ? (CONV_VEC + CONV_THREADS - 1) / CONV_THREADS : 0;
  // bytes landing per stage on the even CTA's `full` (both CTAs' copies of
  // the parts not folded) and on each CTA's raw_full (its folded big parts)
  static constexpr uint32_t PAIR_STAGE_TX =
      2 * ((FOLD_A ? 0 : 2 * A_BYTES) + (FOLD_B ? 0 : 2 * B_BYTES));
  static constexpr uint32_t RAW_TX = (FOLD_A ? A_BYTES : 0) + (FOLD_B ? B_BYTES : 0);
  // arrivals completing `full`: the even producer's, and with a folded part
  // each converter warp of both CTAs
  static constexpr int FULL_COUNT = 1 + 2 * CONV_WARPS;
  static constexpr int REGS_WG0 = 40, REGS_EPI = 232;
  static_assert(BN == 128 || 128 * (REGS_WG0 + 2 * REGS_EPI) <= THREADS * ((65536 / THREADS) & ~7),
                "register split exceeds the launch budget");
};

template <class Cfg>
struct TcPairBars {
  uint32_t base;
  __device__ uint32_t full(uint32_t s) const { return base + 8 * s; }
  __device__ uint32_t empty(uint32_t s) const { return base + 8 * (Cfg::STAGES + s); }
  __device__ uint32_t acc_full(uint32_t b) const { return base + 8 * (2 * Cfg::STAGES + b); }
  __device__ uint32_t acc_empty(uint32_t b) const { return base + 8 * (2 * Cfg::STAGES + 2 + b); }
  __device__ uint32_t drain() const { return base + 8 * (2 * Cfg::STAGES + 4); }
  __device__ uint32_t raw_full(uint32_t s) const { return base + 8 * (2 * Cfg::STAGES + 5 + s); }
};

// Work unit t (p.tiles_m counts 256-row tile rows) -> first row of this
// CTA's 128 rows, the unit's first column, and whether it spans the whole
// tile width (else the half of a tile given by the unit's parity).
template <class Cfg>
__device__ __forceinline__ void pair_tile(const TcParams &p, int t, uint32_t rank, int &m0, int &n0,
                                          bool &whole) {
  whole = t < p.wide_tiles;
  const int u = t - p.wide_tiles;
  const int tile = whole ? t : p.wide_tiles + (u >> 1);
  int tm, tn;
  tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
  m0 = tm * Cfg::BM + 128 * static_cast<int>(rank);
  n0 = tn * Cfg::BN + (whole ? 0 : (u & 1) * (Cfg::BN / 2));
}

// ------------------------------------------------------------------ producer
template <class Cfg>
__device__ __forceinline__ void tcp_produce(const TcParams &p, const CUtensorMap *tmA,
                                            const CUtensorMap *tmB, const CUtensorMap *tmAs,
                                            const CUtensorMap *tmBs, uint32_t sbase,
                                            const TcPairBars<Cfg> &bar, uint32_t rank) {
  uint32_t it = 0;
  bool ok = true;
  for (int t = cluster_id_x(); t < p.num_tiles && ok; t += cluster_count_x()) {
    int m0, n0;
    bool whole;
    pair_tile<Cfg>(p, t, rank, m0, n0, whole);
    // this CTA's half of the unit's op(B) columns (a half-width unit uses
    // the first half of the B_ROWS rows landed)
    const int nb = n0 + (whole ? Cfg::B_ROWS : Cfg::B_ROWS / 2) * static_cast<int>(rank);
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
      const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
      // the stage is free in this CTA once the pair's MMAs on it finished
      if (round > 0 &&
          !wait_parity_bounded(bar.empty(s), (round - 1) & 1, p.wait_budget_ns, p.status)) {
        ok = false;
        break;
      }
      if (rank == 0) {
        if (Cfg::PAIR_STAGE_TX > 0)
          mbar_arrive_expect_tx(bar.full(s), Cfg::PAIR_STAGE_TX);
        else
          mbar_arrive(bar.full(s));
      }
      if constexpr (Cfg::FOLD) mbar_arrive_expect_tx(bar.raw_full(s), Cfg::RAW_TX);
      const uint32_t cfull = map_to_rank(bar.full(s), 0);
      const uint32_t st = sbase + s * Cfg::STAGE_BYTES;
      const int k0 = kt * Cfg::BK;
      if constexpr (Cfg::FOLD_A) {   // the big part only, onto this CTA's raw_full
        tma_load_2d(st + Cfg::A_BIG, tmA, bar.raw_full(s), k0, m0);
      } else {
        tma_load_2d_pair(st + Cfg::A_BIG, tmA, cfull, k0, m0);
        tma_load_2d_pair(st + Cfg::A_SMALL, tmAs, cfull, k0, m0);
      }
      if constexpr (Cfg::FOLD_B) {
        tma_load_2d(st + Cfg::B_BIG, tmB, bar.raw_full(s), k0, nb);
      } else {
        tma_load_2d_pair(st + Cfg::B_BIG, tmB, cfull, k0, nb);
        tma_load_2d_pair(st + Cfg::B_SMALL, tmBs, cfull, k0, nb);
      }
    }
  }
  // On give-up the even CTA lets the copies it counts land (bounded); the
  // cluster barrier at the end keeps the odd CTA alive until then.  Each CTA
  // does the same for the copies onto its own raw_full.
  if (!ok) {
    const uint32_t first = it > Cfg::STAGES ? it - Cfg::STAGES : 0;
    for (uint32_t j = first; j < it; ++j) {
      if (rank == 0)
        wait_parity_bounded(bar.full(j % Cfg::STAGES), (j / Cfg::STAGES) & 1, p.wait_budget_ns,
                            nullptr);
      if constexpr (Cfg::FOLD)
        wait_parity_bounded(bar.raw_full(j % Cfg::STAGES), (j / Cfg::STAGES) & 1, p.wait_budget_ns,
                            nullptr);
    }
  }
}

// ------------------------------------------------------------------ converters
// Converter thread ct's share of stage st: the small parts of this CTA's
// folded big parts, written at the same byte offsets of the small-part tiles
// (an elementwise map keeps the swizzled layout).  All loads are issued
// before the first store.  The stores, made through the generic proxy, are
// fenced for the tensor cores (async proxy), which read them once `full`
// completes.
template <class Cfg>
__device__ __forceinline__ void tcp_convert_stage(uint32_t st, int ct) {
  constexpr int T = Cfg::CONV_THREADS, AV = Cfg::CONV_A_VEC, V = Cfg::CONV_VEC;
  float4 x[Cfg::CONV_PER_THREAD];
#pragma unroll
  for (int j = 0; j < Cfg::CONV_PER_THREAD; ++j) {
    const int i = ct + j * T;
    if (i < V) x[j] = lds128(st + (i < AV ? Cfg::A_BIG + 16 * i : Cfg::B_BIG + 16 * (i - AV)));
  }
#pragma unroll
  for (int j = 0; j < Cfg::CONV_PER_THREAD; ++j) {
    const int i = ct + j * T;
    if (i < V) {
      float4 sm;
      float b0, b1, b2, b3;
      split_pair(x[j].x, x[j].y, b0, b1, sm.x, sm.y);
      split_pair(x[j].z, x[j].w, b2, b3, sm.z, sm.w);
      sts128(st + (i < AV ? Cfg::A_SMALL + 16 * i : Cfg::B_SMALL + 16 * (i - AV)), sm);
    }
  }
  fence_proxy_async_smem();
}

// Wait for stage `it`'s folded big parts, convert this thread's share, and
// count the warp's arrival on the even CTA's `full` (in the even CTA a local
// arrival, whose CTA-scope release covers the MMA thread of the same CTA; in
// the odd one a release at cluster scope).
template <class Cfg>
__device__ __forceinline__ bool tcp_convert_one(const TcParams &p, uint32_t sbase,
                                                const TcPairBars<Cfg> &bar, uint32_t rank,
                                                uint32_t it, int ct, int lane) {
  const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
  if (!wait_parity_bounded(bar.raw_full(s), round & 1, p.wait_budget_ns, p.status)) return false;
  tcp_convert_stage<Cfg>(sbase + s * Cfg::STAGE_BYTES, ct);
  __syncwarp();
  if (lane == 0) {
    if (rank == 0)
      mbar_arrive(bar.full(s));
    else
      mbar_arrive_cluster(map_to_rank(bar.full(s), 0));
  }
  return true;
}

// Warps 2 and 3 at BN = 128: converters only, over every stage.
template <class Cfg>
__device__ __forceinline__ void tcp_convert(const TcParams &p, uint32_t sbase,
                                            const TcPairBars<Cfg> &bar, uint32_t rank, int ct,
                                            int lane) {
  uint32_t it = 0;
  for (int t = cluster_id_x(); t < p.num_tiles; t += cluster_count_x())
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it)
      if (!tcp_convert_one<Cfg>(p, sbase, bar, rank, it, ct, lane)) return;
}

// ------------------------------------------------------------------ MMA issue
// One thread of the even CTA.
template <class Cfg>
__device__ __forceinline__ void tcp_issue(const TcParams &p, uint32_t sbase, uint32_t tmem_base,
                                          const TcPairBars<Cfg> &bar) {
  uint32_t it = 0, chunk_iter = 0;
  bool ok = true;
  for (int t = cluster_id_x(); t < p.num_tiles && ok; t += cluster_count_x()) {
    const uint32_t idesc = t < p.wide_tiles ? Cfg::IDESC : Cfg::IDESC_HALF;
    for (int kc0 = 0; kc0 < p.k_tiles && ok; kc0 += Cfg::CHUNK_KTILES, ++chunk_iter) {
      const uint32_t b = chunk_iter & 1, use = chunk_iter >> 1;
      // both CTAs' epilogues have read this accumulator's previous chunk
      if (use > 0 &&
          !wait_parity_bounded(bar.acc_empty(b), (use - 1) & 1, p.wait_budget_ns, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d = tmem_base + b * Cfg::BN;
      const int kc1 = min(kc0 + Cfg::CHUNK_KTILES, p.k_tiles);
      for (int kt = kc0; kt < kc1; ++kt, ++it) {
        const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
        // with folded parts the peer's converter stores are among what
        // `full` publishes: acquire at cluster scope
        const bool got = Cfg::FOLD ? wait_parity_bounded_cluster(bar.full(s), round & 1,
                                                                 p.wait_budget_ns, p.status)
                                   : wait_parity_bounded(bar.full(s), round & 1, p.wait_budget_ns,
                                                         p.status);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t st = sbase + s * Cfg::STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < Cfg::BK / 8; ++kk) {
          const uint64_t a_big = desc_kmajor_sw128(st + Cfg::A_BIG + kk * 32);
          const uint64_t a_small = desc_kmajor_sw128(st + Cfg::A_SMALL + kk * 32);
          const uint64_t b_big = desc_kmajor_sw128(st + Cfg::B_BIG + kk * 32);
          const uint64_t b_small = desc_kmajor_sw128(st + Cfg::B_SMALL + kk * 32);
          const uint32_t acc = (kt > kc0 || kk > 0) ? 1u : 0u;
          mma_tf32_pair(d, a_small, b_big, idesc, acc);
          mma_tf32_pair(d, a_big, b_small, idesc, 1u);
          mma_tf32_pair(d, a_big, b_big, idesc, 1u);
        }
        mma_commit_pair(bar.empty(s), 0x3);   // frees the stage in both CTAs
      }
      if (!ok) break;
      mma_commit_pair(bar.acc_full(b), 0x3);   // chunk done: both CTAs' epilogues
    }
  }
  // every MMA issued must be complete before tensor memory is released
  mma_commit_pair(bar.drain(), 0x1);
  wait_parity_bounded(bar.drain(), 0, p.wait_budget_ns, nullptr);
}

// ------------------------------------------------------------------ epilogue
// Warp q of epilogue warpgroup `half`: this CTA's tile rows 32q .. 32q+31
// (TMEM lanes), columns 128 * half .. +127.
template <class Cfg>
__device__ __forceinline__ void tcp_epilogue(const TcParams &p, uint32_t tmem_base,
                                             const TcPairBars<Cfg> &bar, uint32_t rank, int q,
                                             int half, int lane) {
  uint32_t chunk_iter = 0;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
  for (int t = cluster_id_x(); t < p.num_tiles; t += cluster_count_x()) {
    int m0, n0;
    bool whole;
    pair_tile<Cfg>(p, t, rank, m0, n0, whole);
    // a half-width unit has no second 128 columns: that warpgroup only keeps
    // the accumulator hand-over in step
    const bool idle = !whole && half > 0;
    float acc[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
    for (int kc0 = 0; kc0 < p.k_tiles; kc0 += Cfg::CHUNK_KTILES, ++chunk_iter) {
      const uint32_t b = chunk_iter & 1, use = chunk_iter >> 1;
      if (!wait_parity_bounded(bar.acc_full(b), use & 1, p.wait_budget_ns, p.status)) return;
      tc_fence_after_sync();
      if (!idle) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + lane_addr + b * Cfg::BN + half * 128 + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(v[j]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(bar.acc_empty(b), 0));
    }
    if (!idle) tc_store_row(p, m0 + 32 * q + lane, n0 + half * 128, acc);
  }
}

// SG_TC_FOLD_LAG: stages converted past the end of an accumulator chunk
// before the epilogue warps hand that chunk over (1 or 2).
#ifndef SG_TC_FOLD_LAG
#define SG_TC_FOLD_LAG 1
#endif

// The epilogue warps with folded parts: converters of every stage, and,
// SG_TC_FOLD_LAG stages after the last stage of each accumulator chunk has
// been converted, the hand-over of that chunk (so the tensor cores have work
// queued while it runs).  The hand-overs follow the same order as in
// tcp_epilogue; the chunk handed over is always one whose stages were all
// converted, so neither job waits on the other's future.
template <class Cfg>
__device__ __forceinline__ void tcp_epilogue_fold(const TcParams &p, uint32_t sbase,
                                                  uint32_t tmem_base, const TcPairBars<Cfg> &bar,
                                                  uint32_t rank, int q, int half, int lane, int ct) {
  const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
  // hand-over cursor: unit td, chunk starting at k-slice kd, chunk count cd
  int td = cluster_id_x(), kd = 0;
  uint32_t cd = 0;
  int m0 = 0, n0 = 0;
  bool whole = true;
  if (td < p.num_tiles) pair_tile<Cfg>(p, td, rank, m0, n0, whole);
  float acc[128];
#pragma unroll
  for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
  auto hand_over = [&]() -> bool {
    const bool idle = !whole && half > 0;   // no second 128 columns
    const uint32_t b = cd & 1, use = cd >> 1;
    if (!wait_parity_bounded(bar.acc_full(b), use & 1, p.wait_budget_ns, p.status)) return false;
    tc_fence_after_sync();
    if (!idle) {
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + b * Cfg::BN + half * 128 + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(v[j]);
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(map_to_rank(bar.acc_empty(b), 0));
    ++cd;
    kd += Cfg::CHUNK_KTILES;
    if (kd >= p.k_tiles) {   // the unit's last chunk: write it, start the next
      if (!idle) tc_store_row(p, m0 + 32 * q + lane, n0 + half * 128, acc);
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      kd = 0;
      td += cluster_count_x();
      if (td < p.num_tiles) pair_tile<Cfg>(p, td, rank, m0, n0, whole);
    }
    return true;
  };
  // last stages of the chunks awaiting hand-over, oldest first (at most
  // SG_TC_FOLD_LAG of them)
  constexpr uint32_t LAG = SG_TC_FOLD_LAG;
  static_assert(LAG >= 1 && LAG <= 2 && LAG < Cfg::STAGES, "hand-over lag of 1 or 2 stages");
  uint32_t it = 0, end0 = 0, end1 = 0;
  int waiting = 0;
  for (int t = cluster_id_x(); t < p.num_tiles; t += cluster_count_x()) {
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
      if (!tcp_convert_one<Cfg>(p, sbase, bar, rank, it, ct, lane)) return;
      while (waiting > 0 && end0 + LAG <= it) {
        if (!hand_over()) return;
        end0 = end1;
        --waiting;
      }
      if ((kt + 1) % Cfg::CHUNK_KTILES == 0 || kt + 1 == p.k_tiles) {
        if (waiting == 0) end0 = it; else end1 = it;
        ++waiting;
      }
    }
  }
  while (waiting-- > 0)
    if (!hand_over()) return;
}

// ------------------------------------------------------------------ kernel
// Launched in clusters of two CTAs; p.tiles_m counts 256-row tile rows,
// p.num_tiles the work units (whole tiles, then column halves: pair_tile).
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc3_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmBs,
                    const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const TcPairBars<Cfg> bar{sbase + Cfg::BAR_OFFSET};
  const uint32_t tmem_slot = sbase + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(bar.full(s), Cfg::FULL_COUNT);
      mbar_init(bar.empty(s), 1);
      if constexpr (Cfg::FOLD) mbar_init(bar.raw_full(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.acc_full(b), 1);
      mbar_init(bar.acc_empty(b), 2 * Cfg::EPILOGUE_WARPS);
    }
    mbar_init(bar.drain(), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmAs);
    tma_prefetch_desc(&tmBs);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  // the peer's copies and arrivals target barriers that must be initialised
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base =
      *reinterpret_cast<volatile uint32_t *>(smem + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8);

  if (warp < 4) {
    if (Cfg::EPILOGUE_GROUPS > 1) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_WG0));
    if (warp == 0) {
      if (lane == 0) tcp_produce<Cfg>(p, &tmA, &tmB, &tmAs, &tmBs, sbase, bar, rank);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0 && rank == 0) tcp_issue<Cfg>(p, sbase, tmem_base, bar);
      __syncwarp();
    } else if constexpr (Cfg::CONV_SIDE_WARPS > 0) {
      tcp_convert<Cfg>(p, sbase, bar, rank, 32 * Cfg::EPILOGUE_WARPS + threadIdx.x - 64, lane);
    }
  } else {
    if (Cfg::EPILOGUE_GROUPS > 1) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_EPI));
    if constexpr (Cfg::FOLD)
      tcp_epilogue_fold<Cfg>(p, sbase, tmem_base, bar, rank, warp & 3, (warp >> 2) - 1, lane,
                             threadIdx.x - 128);
    else
      tcp_epilogue<Cfg>(p, tmem_base, bar, rank, warp & 3, (warp >> 2) - 1, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  // neither CTA releases tensor memory or leaves before the other is done
  cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace sg
