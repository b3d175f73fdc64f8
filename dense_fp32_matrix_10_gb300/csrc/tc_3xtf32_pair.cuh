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
//                `acc_empty` (one arrival per epilogue warp of the pair).
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
template <int BN_>
struct TcPairConfig {
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
  // in the even CTA), drain
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
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
  static constexpr uint32_t PAIR_STAGE_TX = 2 * STAGE_BYTES;   // both CTAs' copies
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
      if (rank == 0) mbar_arrive_expect_tx(bar.full(s), Cfg::PAIR_STAGE_TX);
      const uint32_t cfull = map_to_rank(bar.full(s), 0);
      const uint32_t st = sbase + s * Cfg::STAGE_BYTES;
      const int k0 = kt * Cfg::BK;
      tma_load_2d_pair(st + Cfg::A_BIG, tmA, cfull, k0, m0);
      tma_load_2d_pair(st + Cfg::A_SMALL, tmAs, cfull, k0, m0);
      tma_load_2d_pair(st + Cfg::B_BIG, tmB, cfull, k0, nb);
      tma_load_2d_pair(st + Cfg::B_SMALL, tmBs, cfull, k0, nb);
    }
  }
  // On give-up the even CTA lets the copies it counts land (bounded); the
  // cluster barrier at the end keeps the odd CTA alive until then.
  if (!ok && rank == 0) {
    const uint32_t first = it > Cfg::STAGES ? it - Cfg::STAGES : 0;
    for (uint32_t j = first; j < it; ++j)
      wait_parity_bounded(bar.full(j % Cfg::STAGES), (j / Cfg::STAGES) & 1, p.wait_budget_ns,
                          nullptr);
  }
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
        if (!wait_parity_bounded(bar.full(s), round & 1, p.wait_budget_ns, p.status)) {
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
      mbar_init(bar.full(s), 1);
      mbar_init(bar.empty(s), 1);
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
    }
  } else {
    if (Cfg::EPILOGUE_GROUPS > 1) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_EPI));
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
