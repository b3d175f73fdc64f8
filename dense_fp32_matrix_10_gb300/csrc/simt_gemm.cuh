// simt_gemm.cuh -- CUDA-core (FFMA) single-precision GEMM for sm_103a.
//
// C = alpha * op(A) * op(B) + beta * C, row-major FP32.
//
// Structure (one persistent CTA per SM slot, warp-specialised):
//
//   * a PRODUCER role fills a ring of STAGES shared-memory stages, each holding
//     one BK = 32 slice of the op(A) block tile (BM x 32) and of the op(B) block
//     tile (32 x BN).  Two producers exist:
//       - kTma: one elected thread issues 2-D bulk tensor copies (TMA); the
//         hardware zero-fills everything outside the matrix, and the copy
//         completion is counted in bytes on the stage's "full" mbarrier;
//       - kCpAsync: four warps issue 4-byte cp.async copies (zero-filled
//         outside the matrix) and arrive on the "full" mbarrier when their
//         copies land.  This one takes any alignment and leading dimension.
//   * WARPS_M x WARPS_N MATH warps, each owning a 32 x 64 warp tile, each
//     thread an 8 x 8 register tile of FP32 accumulators.  Per k they read 8
//     op(A) and 8 op(B) values from shared memory as float4s and issue 64 FFMA.
//     A warp releases a stage by arriving on its "empty" mbarrier.
//   * The epilogue writes alpha * acc + beta * C straight from registers,
//     float4-wide where the row is aligned, with row/column predicates on the
//     ragged edges; C is not read when beta == 0.
//
// This is the three-level tiling (grid -> block -> warp -> thread registers)
// and shared-memory reuse of "GPU矩阵乘法优化：共享内存Tiling技术实战" (sections 3.1,
// 7.3) and of the 2D block tiling (b_m, b_n, b_k) of the cloud.baidu.com
// article 9456745, with the register tiling and float4 loads of
// "CUDA矩阵乘法性能优化实战：从朴素内核到寄存器分块与Nsight剖析" (sections 5.2, 5.3)
// taken to 8 x 8.  Its "prefetch the next tile while computing this one" idea
// (the double buffering of the Tiling article, section 3.2) becomes a
// STAGES-deep mbarrier ring filled by a dedicated producer; the +1 padding that
// those pages use against bank conflicts (Tiling article 4.1; optimisation
// article 3.3) becomes the TMA 128-byte swizzle on the k-contiguous tiles.
//
// Shared-memory layouts of one stage (all FP32):
//   op(A) tile, A stored M x K (k contiguous, "K-major"):  [BM rows][32 k],
//       128 B per row, 16-byte chunk j of row m stored at chunk j ^ (m & 7).
//   op(A) tile, A stored K x M (m contiguous, "MN-major"): [32 k][BM m], dense.
//   op(B) tile, B stored K x N (n contiguous, "MN-major"): [32 k][BN n], dense.
//   op(B) tile, B stored N x K (k contiguous, "K-major"):  [BN rows][32 k],
//       same swizzle as above.
//
// Thread -> output mapping inside a 32 x 8TN warp tile (lane = 8 * tm + tn,
// tm in 0..3, tn in 0..7; thread tile 8 x TN, TN = 8 or 16), chosen so that
// the eight lanes of each quarter-warp read distinct banks or the same word:
//   rows: MN-major A: {4tm .. 4tm+3, 16+4tm .. 16+4tm+3};  K-major A: tm + 4r.
//   cols: MN-major B: 4tn + 32h + {0..3}, h < TN/4;        K-major B: tn + 8c.
// Every LDS.128 of a warp takes four shared-memory wavefronts whatever the
// broadcast, so a thread loads (8 + TN) floats per k for 8*TN FMAs: TN = 16
// keeps shared-memory traffic at 75% of the FMA rate (TN = 8: 100%).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace sg {

enum Producer : int { kTma = 0, kCpAsync = 1 };

struct SimtParams {
  const float *A;
  const float *B;
  float *C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  float alpha, beta;
  int tiles_m, tiles_n, k_tiles, num_tiles;
  int group_m;           // tile-rows per raster group (L2 reuse)
  int c_vec4;            // ldc % 4 == 0 and C 16-byte aligned
  uint64_t wait_budget_ns;
  int *status;
  // Work split (stream-K).  Tiles [0, dp_tiles) are whole-k units handed out
  // round-robin; the k-iterations of tiles [dp_tiles, num_tiles) are divided
  // evenly over the grid: CTA g takes iterations [g*sk_iters/G, (g+1)*sk_iters/G)
  // of that region.  A segment that does not cover a whole tile writes its raw
  // partial sums to workspace slot 2g (the CTA's first segment) or 2g+1 (its
  // last); sk_fixup_kernel adds them in k order and applies alpha/beta.
  int dp_tiles;
  int64_t sk_iters;      // (num_tiles - dp_tiles) * k_tiles
  float *workspace;      // 2 * gridDim.x slots of BM * BN floats
  // Strided batch: product b uses A + b*strideA, B + b*strideB, C + b*strideC
  // (elements; a zero stride shares one operand across the batch).  Tiles are
  // numbered batch-major: num_tiles = batch * tiles_per_batch.  With the TMA
  // producer a strided operand's tensor map has a third (batch) dimension.
  int tiles_per_batch;
  int64_t strideA, strideB, strideC;
  int a_map3d, b_map3d;
  // In-kernel fixup: one arrival counter per stream-K tile (zero between
  // launches).  Every segment stores its partial and counts itself in; the
  // CTA that arrives last adds the tile's partials in k order and writes C.
  // Null: sk_fixup_kernel does that in a second launch.
  int *sk_count = nullptr;
  // Cluster split-K (csk = S > 1): the kernel is launched in clusters of S
  // CTAs along x, grid = S * num_tiles, and cluster c computes tile c with
  // its k-tiles divided over the S CTAs (rank r takes [r*KT/S, (r+1)*KT/S)).
  // Each CTA leaves its partial tile in its own shared memory; after a
  // cluster-wide handshake CTA r adds rows [r*BM/S, (r+1)*BM/S) of the S
  // partials, in rank order, through distributed shared memory and writes C.
  // No workspace, no second launch.  0: off.
  int csk = 0;
  // C written by TMA stores (EPI_TMA kernels; beta == 0 and C addressable by
  // the tmC tensor map: 2-D, or 3-D with the batch stride)
  int c_tma = 0;
  // beta != 0 and C addressable by tmC (1: 2-D, 2: 3-D): the TMA producer
  // prefetches each C tile into L2 before the epilogue reads it
  int c_pref = 0;
};

// Batch index and (tile_m, tile_n) of linear tile t.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn);
__device__ __forceinline__ void unit_coords(const SimtParams &p, int t, int &b, int &tm, int &tn) {
  b = t / p.tiles_per_batch;
  tile_coords(t - b * p.tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
}

// One unit of work: k-tiles [k0, k1) of tile `tile`; slot -1 writes C,
// kCskSlot is a cluster split-K share, slot >= 0 a stream-K partial.
struct WorkUnit {
  int tile, k0, k1, slot;
};
constexpr int kCskSlot = -2;

// Visits this CTA's units in order; f returns false to stop early.  Every
// role of the CTA walks the same sequence.
template <bool CSK, class F>
__device__ __forceinline__ void for_each_unit(const SimtParams &p, F &&f) {
  if constexpr (CSK) {   // cluster split-K: one share of one tile (cluster dims (S, 1, 1))
    const int S = p.csk, r = static_cast<int>(blockIdx.x) % S;
    const int k0 = static_cast<int>(static_cast<int64_t>(r) * p.k_tiles / S);
    const int k1 = static_cast<int>(static_cast<int64_t>(r + 1) * p.k_tiles / S);
    f(WorkUnit{static_cast<int>(blockIdx.x) / S, k0, k1, kCskSlot});
    return;
  }
  for (int t = blockIdx.x; t < p.dp_tiles; t += gridDim.x)
    if (!f(WorkUnit{t, 0, p.k_tiles, -1})) return;
  if (p.sk_iters > 0) {
    const int64_t g = blockIdx.x, G = gridDim.x;
    const int64_t first = g * p.sk_iters / G, end = (g + 1) * p.sk_iters / G;
    for (int64_t it = first; it < end;) {
      const int ts = static_cast<int>(it / p.k_tiles);
      const int k0 = static_cast<int>(it - static_cast<int64_t>(ts) * p.k_tiles);
      const int64_t rest = static_cast<int64_t>(k0) + (end - it);
      const int k1 = rest < p.k_tiles ? static_cast<int>(rest) : p.k_tiles;
      const bool whole = (k0 == 0 && k1 == p.k_tiles);
      if (!f(WorkUnit{p.dp_tiles + ts, k0, k1, whole ? -1 : static_cast<int>(2 * g + (it == first ? 0 : 1))}))
        return;
      it += k1 - k0;
    }
  }
}

// Calls f(i, slot) for the CTA segments covering stream-K tile ts (its index
// within the stream-K region) in increasing k order (i = 0, 1, ...), with the
// workspace slot each stored its partial in (slot 2g: CTA g's first unit,
// 2g + 1: its last); returns their number.  G = the main grid.
template <class F>
__device__ __forceinline__ int sk_for_each_segment(const SimtParams &p, int64_t G, int ts, F &&f) {
  const int64_t KT = p.k_tiles, S = p.sk_iters;
  const int64_t it0 = static_cast<int64_t>(ts) * KT, it1 = it0 + KT;
  int64_t g = it0 * G / S;
  while (g + 1 < G && (g + 1) * S / G <= it0) ++g;
  while (g > 0 && g * S / G > it0) --g;
  int n = 0;
  for (; g < G; ++g) {
    const int64_t a = g * S / G, b = (g + 1) * S / G;
    if (a >= it1) break;
    if ((a > it0 ? a : it0) >= (b < it1 ? b : it1)) continue;  // empty segment
    f(n, static_cast<int>(2 * g + (a >= it0 ? 0 : 1)));
    ++n;
  }
  return n;
}

// SG_SIMT_PREFETCH_C    the TMA producer asks L2 for a unit's C tile (beta != 0)
//                        when it issues the loads of the unit's k-slice this
//                        many before the last (0: never).
#ifndef SG_SIMT_PREFETCH_C
#define SG_SIMT_PREFETCH_C 2
#endif

// SG_SIMT_TRANSPOSERS  producer warps (1..3) that share the A transpose;
// SG_SIMT_TRANSPOSER_REGS their registers per thread (the math warps get the
// rest of the launch budget); SG_SIMT_TRANSPOSE_UNROLL rows in flight.
#ifndef SG_SIMT_TRANSPOSERS
#define SG_SIMT_TRANSPOSERS 3
#endif
#ifndef SG_SIMT_TRANSPOSER_REGS
#define SG_SIMT_TRANSPOSER_REGS 56
#endif
#ifndef SG_SIMT_TRANSPOSE_UNROLL
#define SG_SIMT_TRANSPOSE_UNROLL 4
#endif
// SG_SIMT_CPASYNC_REGS: registers per thread of the cp.async producer warps;
// SG_SIMT_CPASYNC_UNROLL: copies each of them unrolls.
#ifndef SG_SIMT_CPASYNC_REGS
#define SG_SIMT_CPASYNC_REGS 40
#endif
#ifndef SG_SIMT_CPASYNC_UNROLL
#define SG_SIMT_CPASYNC_UNROLL 2
#endif

template <int WARPS_M_, int WARPS_N_, bool A_KMAJOR_, bool B_KMAJOR_, int STAGES_, int PRODUCER_,
          int TN_ = 8, bool A_TRANS_ = false, bool CSK_ = false>
struct SimtConfig {
  // CSK: the cluster split-K form (SimtParams::csk); a separate
  // instantiation, so that the other kernels carry none of its code.  Its
  // partial tile is staged in the stage ring.
  static constexpr bool CSK = CSK_;
  static constexpr int WARPS_M = WARPS_M_;
  static constexpr int WARPS_N = WARPS_N_;
  static constexpr bool A_KMAJOR = A_KMAJOR_;  // layout of A in global memory
  static constexpr bool B_KMAJOR = B_KMAJOR_;
  static constexpr int STAGES = STAGES_;
  static constexpr int PRODUCER = PRODUCER_;
  // A_TRANS: the TMA lands a k-contiguous A tile in a raw ring and producer
  // warps rewrite it m-contiguous into the stage.
  static constexpr bool A_TRANS = A_TRANS_;
  static_assert(!A_TRANS || (A_KMAJOR && PRODUCER == kTma), "A transpose: k-contiguous A, TMA");
  static constexpr bool A_SMEM_KMAJOR = A_KMAJOR && !A_TRANS;  // layout the math warps read
  // Thread tile 8 x TN (TN = 8 or 16); warp tile 32 x 8*TN; lanes 4 x 8.
  static constexpr int TN = TN_;
  static constexpr int WN = 8 * TN;
  static constexpr int BM = 32 * WARPS_M;
  static constexpr int BN = WN * WARPS_N;
  static_assert(TN == 8 || (TN == 16 && !B_KMAJOR), "16-wide thread tiles need n-contiguous op(B)");
  static constexpr int BK = 32;
  static constexpr int MATH_WARPS = WARPS_M * WARPS_N;
  static constexpr int MATH_THREADS = 32 * MATH_WARPS;
  // The producer role is a whole warpgroup so that setmaxnreg can hand its
  // registers to the math warpgroups (register files are per SM
  // sub-partition: a 9-warp CTA would cap every thread at 168 registers).
  static constexpr int PRODUCER_WARPS = 4;
  static constexpr int PRODUCER_THREADS = 32 * PRODUCER_WARPS;
  static constexpr int TRANSPOSER_WARPS = SG_SIMT_TRANSPOSERS;  // producer warps 1.. when A_TRANS
  static constexpr int THREADS = MATH_THREADS + PRODUCER_THREADS;
  static constexpr int MIN_CTAS = (MATH_WARPS == 8) ? 1 : 2;  // CTAs per SM
  // Per-thread registers after the split; launch budget is
  // THREADS * (65536 / (THREADS * MIN_CTAS)) rounded down to 8.
  // The bare TMA producer needs few registers; the cp.async producer and the
  // transposing producer warps need more.
  static constexpr bool LEAN_PRODUCER = (PRODUCER == kTma) && !A_TRANS;
  static constexpr int LAUNCH_REGS = (65536 / (THREADS * MIN_CTAS)) & ~7;
  static constexpr int PRODUCER_REGS =
      LEAN_PRODUCER ? 24 : (A_TRANS ? SG_SIMT_TRANSPOSER_REGS : SG_SIMT_CPASYNC_REGS);
  static constexpr int MATH_REGS_FIT =
      ((THREADS * LAUNCH_REGS - PRODUCER_THREADS * PRODUCER_REGS) / MATH_THREADS) & ~7;
  static constexpr int MATH_REGS = MATH_REGS_FIT < 240 ? MATH_REGS_FIT : 240;
  static_assert(MATH_WARPS % 4 == 0, "math role must be whole warpgroups");
  static_assert(PRODUCER_THREADS * PRODUCER_REGS + MATH_THREADS * MATH_REGS <=
                    THREADS * ((65536 / (THREADS * MIN_CTAS)) & ~7),
                "register split exceeds the launch budget");
  static constexpr int A_STAGE_BYTES = BM * BK * 4;
  static constexpr int B_STAGE_BYTES = BN * BK * 4;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  // stages first (1024-byte aligned for the 128 B swizzle), then the raw A
  // ring (A_TRANS), then the barriers
  static constexpr int RAW_A_STAGES = A_TRANS ? 2 : 0;
  static constexpr int RAW_A_OFFSET = STAGES * STAGE_BYTES;
  // EPI_TMA: the 128 x 128 TMA kernels can stage a finished tile in shared
  // memory (four 32-column boxes, 128-byte swizzle) and write it to C with
  // TMA stores, so the math warps go on to the next tile while it drains.
  // Not the NT kernel (A transposed in shared memory, B k-contiguous), whose
  // transposing warps already load shared memory heavily: there it lost
  // (GB300, 96 x 512x512x64: NT 36.3 -> 35.6 TFLOP/s, against NN 36.3 ->
  // 39.1, TN 38.2 -> 40.6, TT 37.3 -> 38.9).
  static constexpr bool EPI_TMA =
      (PRODUCER == kTma) && (MATH_WARPS == 8) && (TN == 8) && !(A_TRANS && B_KMAJOR);
  static constexpr int STAGING_OFFSET = RAW_A_OFFSET + RAW_A_STAGES * A_STAGE_BYTES;
  static constexpr int STAGING_BYTES = EPI_TMA ? BM * BN * 4 : 0;
  static constexpr int BAR_OFFSET = STAGING_OFFSET + STAGING_BYTES;
  // full[STAGES], empty[STAGES], raw_full[2], raw_empty[2]
  static constexpr int SMEM_BYTES = BAR_OFFSET + (2 * STAGES + 4) * 8 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
  // arrivals that complete a stage's `full` barrier
  static constexpr int FULL_COUNT =
      (PRODUCER == kTma) ? (A_TRANS ? 1 + TRANSPOSER_WARPS : 1) : PRODUCER_THREADS;
  static_assert(BM <= 256 && BN <= 256, "TMA box extent is at most 256");
  static_assert(!CSK || BM * BN * 4 <= STAGES * STAGE_BYTES, "the cluster split-K partial fits the ring");
  static_assert(A_STAGE_BYTES % 1024 == 0 && B_STAGE_BYTES % 1024 == 0, "swizzle atom alignment");
};

// Linear tile index -> (tile_m, tile_n), grouped so that consecutive tiles
// share op(A) row-blocks in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int rows_here = min(tiles_m - first_m, group_m);
  const int r = t - g * per_group;
  tm = first_m + r % rows_here;
  tn = r / rows_here;
}

// Byte offset of element (row, k) in a [rows][32] swizzled tile.
__device__ __forceinline__ uint32_t kmajor_offset(int row, int k) {
  return static_cast<uint32_t>(row) * 128u +
         ((static_cast<uint32_t>((k >> 2) ^ (row & 7))) << 4) + (static_cast<uint32_t>(k & 3) << 2);
}

// ------------------------------------------------------------------ producer
// TMA prefetch of one box of C into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int32_t c0, int32_t c1,
                                                   int32_t c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

template <class Cfg>
__device__ __forceinline__ void produce_tma(const SimtParams &p, const CUtensorMap *tmA,
                                            const CUtensorMap *tmB, const CUtensorMap *tmC,
                                            uint32_t smem_base, uint32_t full0, uint32_t empty0,
                                            uint32_t raw_full0, uint32_t raw_empty0, bool &ok) {
  uint32_t it = 0;        // k-slices whose stage copies are issued
  uint32_t raw_it = 0;    // k-slices whose raw A copies are issued
  for_each_unit<Cfg::CSK>(p, [&](const WorkUnit &u) {
    int bi, tm, tn;
    unit_coords(p, u.tile, bi, tm, tn);
    const int m0 = tm * Cfg::BM, n0 = tn * Cfg::BN;
    // beta != 0: the epilogue will read this tile of C (the unit writes C, or
    // may finish its split tile in-kernel); ask L2 for it a little ahead
    const int pf_kt = (SG_SIMT_PREFETCH_C > 0 && p.c_pref && (u.slot < 0 || p.sk_count != nullptr))
                          ? (u.k1 - SG_SIMT_PREFETCH_C > u.k0 ? u.k1 - SG_SIMT_PREFETCH_C : u.k0)
                          : -1;
    for (int kt = u.k0; kt < u.k1; ++kt) {
      const uint32_t s = it % Cfg::STAGES;
      const uint32_t round = it / Cfg::STAGES;
      const int k0 = kt * Cfg::BK;
      if (kt == pf_kt) {
        for (int j = 0; j < Cfg::BN / 32 && n0 + 32 * j < p.N; ++j) {
          if (p.c_pref == 2)
            tma_prefetch_l2_3d(tmC, n0 + 32 * j, m0, bi);
          else
            tma_prefetch_l2_2d(tmC, n0 + 32 * j, m0);
        }
      }
      if (Cfg::A_TRANS) {  // A: raw k-contiguous tile into the raw ring
        const uint32_t r = raw_it % 2, rr = raw_it / 2;
        if (rr > 0 &&
            !wait_parity_bounded(raw_empty0 + 8 * r, (rr - 1) & 1, p.wait_budget_ns, p.status)) {
          ok = false;
          return false;
        }
        mbar_arrive_expect_tx(raw_full0 + 8 * r, Cfg::A_STAGE_BYTES);
        const uint32_t raw_dst = smem_base + Cfg::RAW_A_OFFSET + r * Cfg::A_STAGE_BYTES;
        if (p.a_map3d)
          tma_load_3d(raw_dst, tmA, raw_full0 + 8 * r, k0, m0, bi);
        else
          tma_load_2d(raw_dst, tmA, raw_full0 + 8 * r, k0, m0);
        ++raw_it;
      }
      if (round > 0 &&
          !wait_parity_bounded(empty0 + 8 * s, (round - 1) & 1, p.wait_budget_ns, p.status)) {
        ok = false;
        return false;
      }
      const uint32_t full = full0 + 8 * s;
      const uint32_t a_dst = smem_base + s * Cfg::STAGE_BYTES;
      const uint32_t b_dst = a_dst + Cfg::A_STAGE_BYTES;
      mbar_arrive_expect_tx(full, Cfg::A_TRANS ? Cfg::B_STAGE_BYTES : Cfg::STAGE_BYTES);
      if (!Cfg::A_TRANS) {
        const int c0 = Cfg::A_KMAJOR ? k0 : m0, c1 = Cfg::A_KMAJOR ? m0 : k0;
        if (p.a_map3d)
          tma_load_3d(a_dst, tmA, full, c0, c1, bi);
        else
          tma_load_2d(a_dst, tmA, full, c0, c1);
      }
      {
        const int c0 = Cfg::B_KMAJOR ? k0 : n0, c1 = Cfg::B_KMAJOR ? n0 : k0;
        if (p.b_map3d)
          tma_load_3d(b_dst, tmB, full, c0, c1, bi);
        else
          tma_load_2d(b_dst, tmB, full, c0, c1);
      }
      ++it;
    }
    return true;
  });
  if (!ok) {
    // Let the copies already issued land before the CTA can end.
    const uint32_t first = it > Cfg::STAGES ? it - Cfg::STAGES : 0;
    for (uint32_t j = first; j < it; ++j)
      wait_parity_bounded(full0 + 8 * (j % Cfg::STAGES), (j / Cfg::STAGES) & 1,
                          p.wait_budget_ns, nullptr);
    const uint32_t rfirst = raw_it > 2 ? raw_it - 2 : 0;
    for (uint32_t j = rfirst; j < raw_it; ++j)
      wait_parity_bounded(raw_full0 + 8 * (j % 2), (j / 2) & 1, p.wait_budget_ns, nullptr);
  }
}

// Producer warps 1..3 when A_TRANS: raw k-contiguous A tile (128-byte rows,
// 128 B swizzle) -> m-contiguous [32 k][BM m] in the stage.  Lane l handles
// row m = 32*mb + l: its LDS.128 of chunk c and the 4 stores of the quarter
// warp both touch every bank once.
template <class Cfg>
__device__ __forceinline__ void transpose_a(const SimtParams &p, unsigned char *smem,
                                            uint32_t full0, uint32_t empty0, uint32_t raw_full0,
                                            uint32_t raw_empty0, int tw, int lane, bool &ok) {
  constexpr int BM = Cfg::BM, ITEMS = (BM / 32) * 8;
  uint32_t it = 0;
  for_each_unit<Cfg::CSK>(p, [&](const WorkUnit &u) {
    for (int kt = u.k0; kt < u.k1; ++kt, ++it) {
      const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
      const uint32_t r = it % 2, rr = it / 2;
      if (!wait_parity_bounded(raw_full0 + 8 * r, rr & 1, p.wait_budget_ns, p.status) ||
          (round > 0 &&
           !wait_parity_bounded(empty0 + 8 * s, (round - 1) & 1, p.wait_budget_ns, p.status))) {
        ok = false;
        return false;
      }
      const unsigned char *raw = smem + Cfg::RAW_A_OFFSET + r * Cfg::A_STAGE_BYTES;
      float *dst = reinterpret_cast<float *>(smem + s * Cfg::STAGE_BYTES);
      constexpr int UNROLL = SG_SIMT_TRANSPOSE_UNROLL;
#pragma unroll UNROLL
      for (int item = tw; item < ITEMS; item += Cfg::TRANSPOSER_WARPS) {
        const int c = item & 7, m = (item >> 3) * 32 + lane;
        if (!SG_CHECK(m < BM && (4 * c + 3) * BM + m < Cfg::BK * BM, p.status)) continue;
        const float4 v = *reinterpret_cast<const float4 *>(raw + m * 128 + ((c ^ (m & 7)) << 4));
        dst[(4 * c + 0) * BM + m] = v.x;
        dst[(4 * c + 1) * BM + m] = v.y;
        dst[(4 * c + 2) * BM + m] = v.z;
        dst[(4 * c + 3) * BM + m] = v.w;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(full0 + 8 * s);
        mbar_arrive(raw_empty0 + 8 * r);
      }
    }
    return true;
  });
}

template <class Cfg>
__device__ __forceinline__ void produce_cpasync(const SimtParams &p, uint32_t smem_base,
                                                uint32_t full0, uint32_t empty0, int ptid,
                                                bool &ok) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK;
  constexpr int PT = Cfg::PRODUCER_THREADS;
  constexpr int UNROLL = SG_SIMT_CPASYNC_UNROLL;
  uint32_t it = 0;
  for_each_unit<Cfg::CSK>(p, [&](const WorkUnit &u) {
    int bi, tm, tn;
    unit_coords(p, u.tile, bi, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const float *Ab = p.A + static_cast<int64_t>(bi) * p.strideA;
    const float *Bb = p.B + static_cast<int64_t>(bi) * p.strideB;
    for (int kt = u.k0; kt < u.k1; ++kt, ++it) {
      const uint32_t s = it % Cfg::STAGES;
      const uint32_t round = it / Cfg::STAGES;
      if (round > 0 &&
          !wait_parity_bounded(empty0 + 8 * s, (round - 1) & 1, p.wait_budget_ns, p.status)) {
        ok = false;
        return false;
      }
      const uint32_t a_dst = smem_base + s * Cfg::STAGE_BYTES;
      const uint32_t b_dst = a_dst + Cfg::A_STAGE_BYTES;
      const int k0 = kt * BK;
      // op(A) tile: BM x 32 elements
#pragma unroll UNROLL
      for (int e = ptid; e < BM * BK; e += PT) {
        int m, k;
        uint32_t off;
        if (Cfg::A_KMAJOR) {  // consecutive threads walk k inside one row
          m = e / BK;
          k = e % BK;
          off = kmajor_offset(m, k);
        } else {  // consecutive threads walk m inside one k-row
          k = e / BM;
          m = e % BM;
          off = static_cast<uint32_t>(k * BM + m) * 4u;
        }
        const int gm = m0 + m, gk = k0 + k;
        const bool in = gm < p.M && gk < p.K;
        const float *src = p.A;
        if (in) src = Cfg::A_KMAJOR ? Ab + static_cast<int64_t>(gm) * p.lda + gk
                                    : Ab + static_cast<int64_t>(gk) * p.lda + gm;
        if (SG_CHECK(off + 4 <= static_cast<uint32_t>(Cfg::A_STAGE_BYTES) && m < BM && k < BK, p.status))
          cp_async_4(a_dst + off, src, in ? 4u : 0u);
      }
      // op(B) tile: 32 x BN elements
#pragma unroll UNROLL
      for (int e = ptid; e < BN * BK; e += PT) {
        int n, k;
        uint32_t off;
        if (Cfg::B_KMAJOR) {
          n = e / BK;
          k = e % BK;
          off = kmajor_offset(n, k);
        } else {
          k = e / BN;
          n = e % BN;
          off = static_cast<uint32_t>(k * BN + n) * 4u;
        }
        const int gn = n0 + n, gk = k0 + k;
        const bool in = gn < p.N && gk < p.K;
        const float *src = p.B;
        if (in) src = Cfg::B_KMAJOR ? Bb + static_cast<int64_t>(gn) * p.ldb + gk
                                    : Bb + static_cast<int64_t>(gk) * p.ldb + gn;
        if (SG_CHECK(off + 4 <= static_cast<uint32_t>(Cfg::B_STAGE_BYTES) && n < BN && k < BK, p.status))
          cp_async_4(b_dst + off, src, in ? 4u : 0u);
      }
      cp_async_mbar_arrive_noinc(full0 + 8 * s);
    }
    return true;
  });
  // Do not leave while this thread's copies are still in flight.
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------ consumer
template <class Cfg>
__device__ __forceinline__ int thread_row(int tm, int r) {
  return Cfg::A_SMEM_KMAJOR ? (tm + 4 * r) : ((r < 4) ? (4 * tm + r) : (16 + 4 * tm + (r - 4)));
}
template <class Cfg>
__device__ __forceinline__ int thread_col(int tn, int c) {
  return Cfg::B_KMAJOR ? (tn + 8 * c) : (32 * (c >> 2) + 4 * tn + (c & 3));
}

// Inner-product options (compile-time):
//   SG_SIMT_FFMA2     1: packed FP32 FMA (__ffma2_rn: two FMAs per instruction,
//                        each rounded like fmaf) where the layout gives natural
//                        register pairs; 0: scalar fmaf everywhere.
//   SG_SIMT_KC_UNROLL, SG_SIMT_KC_UNROLL_WIDE
//                     how many 4-k chunks of a 32-k stage are unrolled (1..8)
//                     for 8 x 8 and for 8 x 16 thread tiles (the wider tile
//                     holds 128 accumulators and spills when unrolled deeper).
#ifndef SG_SIMT_FFMA2
#define SG_SIMT_FFMA2 1
#endif
#ifndef SG_SIMT_KC_UNROLL
#define SG_SIMT_KC_UNROLL 8
#endif
#ifndef SG_SIMT_KC_UNROLL_WIDE
#define SG_SIMT_KC_UNROLL_WIDE 1
#endif
// SG_SIMT_KA_PAIR_ROWS: k values of an m-contiguous op(A) held at once when
// op(B) is k-contiguous (the row-paired FFMA2 form): each k costs the same two
// LDS.128 whatever the grouping; fewer held values leave room for op(B)'s
// 4 k x 8 column fragment.
#ifndef SG_SIMT_KA_PAIR_ROWS
#define SG_SIMT_KA_PAIR_ROWS 4
#endif

// SG_SIMT_TRANSPOSE_A  1: with the TMA producer, a k-contiguous op(A) tile is
//                        rewritten m-contiguous in shared memory by three
//                        producer warps, so the math warps always read A as
//                        [k][m] (conflict-free float4 rows, fewer registers,
//                        the 8 x 16 tile becomes usable); 0: math warps read
//                        the swizzled k-contiguous tile directly.
#ifndef SG_SIMT_TRANSPOSE_A
#define SG_SIMT_TRANSPOSE_A 1
#endif

// SG_SIMT_KC_UNROLL_CPASYNC: the unroll of the kernels fed by cp.async.
// Fully unrolled they spilled 8-140 bytes; not unrolled (and with the
// producer's copies unrolled by 2) none spills and all are faster (GB300,
// graph replays, 1024^3 forced to cp.async: NN 98.0 -> 92.0 us, NT 117.3 ->
// 112.1, TN 98.6 -> 90.2, TT 98.8 -> 92.8).  The TMA kernels stay fully
// unrolled: for those reading a k-contiguous op(B) tile the spill-free
// forms measured slower (unroll 1: 1024^3 TT 50.9 -> 52.7 us, NT 53.0 ->
// 55.0; 4096^3 TT 2259 -> 2359 us), so their 32-80 spilled bytes are kept.
#ifndef SG_SIMT_KC_UNROLL_CPASYNC
#define SG_SIMT_KC_UNROLL_CPASYNC 1
#endif
// SG_SIMT_KC_UNROLL_BK: the unroll of the TMA kernels whose op(B) tile is
// k-contiguous (op(B)'s 4 k x 8 column fragment is held per chunk).
#ifndef SG_SIMT_KC_UNROLL_BK
#define SG_SIMT_KC_UNROLL_BK 8
#endif
template <class Cfg>
__host__ __device__ constexpr int kc_unroll() {
  return Cfg::TN == 16 ? SG_SIMT_KC_UNROLL_WIDE
         : Cfg::PRODUCER == kCpAsync ? SG_SIMT_KC_UNROLL_CPASYNC
         : Cfg::B_KMAJOR             ? SG_SIMT_KC_UNROLL_BK
                                     : SG_SIMT_KC_UNROLL;
}

// How the 64 accumulators of a thread are packed into 32 float2 and updated.
// A packed FMA needs both multiplicands as register pairs; one of them is a
// broadcast (x, x), the other must be two consecutive floats of one LDS.128:
//   kPairCols: (row r, cols c, c+1) pairs; needs op(B) n-contiguous in smem;
//   kPairRows: (rows r, r+1, col c) pairs; needs op(A) m-contiguous in smem;
//   kScalar:   both operands k-contiguous -- no natural pair; scalar FFMA.
enum AccMode : int { kPairCols = 0, kPairRows = 1, kScalar = 2 };

template <class Cfg>
__device__ __host__ constexpr int acc_mode() {
  return !SG_SIMT_FFMA2 ? kScalar
                        : (!Cfg::B_KMAJOR ? kPairCols : (!Cfg::A_SMEM_KMAJOR ? kPairRows : kScalar));
}

// 8 x TN accumulators packed as 4*TN float2.
template <class Cfg>
using AccT = float2[4 * Cfg::TN];

// Storage slot and half of output (r, c) of the thread's 8 x TN tile
// (kPairRows is only used with TN = 8).
template <int MODE, int TN, class A>
__device__ __forceinline__ float &acc_ref(A &acc, int r, int c) {
  if (MODE == kPairRows) return (r & 1) ? acc[(r >> 1) * TN + c].y : acc[(r >> 1) * TN + c].x;
  return (c & 1) ? acc[r * (TN / 2) + (c >> 1)].y : acc[r * (TN / 2) + (c >> 1)].x;
}
template <int MODE, int TN, class A>
__device__ __forceinline__ float acc_get(const A &acc, int r, int c) {
  if (MODE == kPairRows) return (r & 1) ? acc[(r >> 1) * TN + c].y : acc[(r >> 1) * TN + c].x;
  return (c & 1) ? acc[r * (TN / 2) + (c >> 1)].y : acc[r * (TN / 2) + (c >> 1)].x;
}

template <class Cfg>
__device__ __forceinline__ void mma_stage(AccT<Cfg> &acc, const char *a_stage, const char *b_stage,
                                          int wm, int wn, int tm, int tn, int *status) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, TN = Cfg::TN;
  constexpr int MODE = acc_mode<Cfg>();
  // Per-thread base pointers inside the stage.
  const char *a_base;
  const char *b_base;
  if (Cfg::A_SMEM_KMAJOR)
    a_base = a_stage + (wm * 32 + tm) * 128;  // row tm + 4r -> + r * 512
  else
    a_base = a_stage + (wm * 32 + 4 * tm) * 4;  // + k * BM * 4, + 64 for rows 16..
  if (Cfg::B_KMAJOR)
    b_base = b_stage + (wn * Cfg::WN + tn) * 128;  // row tn + 8c -> + c * 1024
  else
    b_base = b_stage + (wn * Cfg::WN + 4 * tn) * 4;  // + k * BN * 4, + 128 per column group

  if constexpr (SGEMM_DEBUG_BOUNDS) {
    // the farthest byte each operand's reads reach in this stage
    const int a_last = Cfg::A_SMEM_KMAJOR ? (wm * 32 + tm + 28) * 128 + 128
                                          : ((31 * BM + wm * 32 + 4 * tm + 16) + 4) * 4;
    const int b_last = Cfg::B_KMAJOR ? (wn * Cfg::WN + tn + 8 * (TN - 1)) * 128 + 128
                                     : ((31 * BN + wn * Cfg::WN + 4 * tn + 32 * (TN / 4 - 1)) + 4) * 4;
    if (!SG_CHECK(a_last <= Cfg::A_STAGE_BYTES && b_last <= Cfg::B_STAGE_BYTES, status)) return;
  }
  constexpr int KC_UNROLL = kc_unroll<Cfg>();
#pragma unroll KC_UNROLL
  for (int kc = 0; kc < 8; ++kc) {  // 4 k per chunk
    float bk[4][8];  // k-contiguous op(B) (TN == 8): bk[kk][c]
    if (Cfg::B_KMAJOR) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        // row = wn*64 + tn + 8c: (row & 7) = tn
        const int sw = (kc ^ tn) << 4;
        const float4 v = *reinterpret_cast<const float4 *>(b_base + c * 1024 + sw);
        bk[0][c] = v.x; bk[1][c] = v.y; bk[2][c] = v.z; bk[3][c] = v.w;
      }
    }
    // op(A) values are loaded KA k at a time (k-contiguous: one LDS of KA floats
    // per row; the wavefront count is the same for KA = 2 and 4, KA = 2 holds
    // half the registers, which the 8 x 16 tile needs).
    constexpr int KA = (TN == 16) ? 2 : (MODE == kPairRows ? SG_SIMT_KA_PAIR_ROWS : 4);
#pragma unroll
    for (int kg = 0; kg < 4 / KA; ++kg) {
      float a[8][KA];  // a[r][j] = op(A)(row r, k = kc*4 + kg*KA + j)
      if (Cfg::A_SMEM_KMAJOR) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          // row = wm*32 + tm + 4r: (row & 7) = tm | 4*(r&1)
          const char *src = a_base + r * 512 + ((kc ^ (tm | ((r & 1) << 2))) << 4) + kg * KA * 4;
          if constexpr (KA == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            a[r][0] = v.x; a[r][1] = v.y; a[r][2] = v.z; a[r][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2 *>(src);
            a[r][0] = v.x; a[r][1] = v.y;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < KA; ++j) {
          const char *row = a_base + (kc * 4 + kg * KA + j) * BM * 4;
          const float4 v0 = *reinterpret_cast<const float4 *>(row);
          const float4 v1 = *reinterpret_cast<const float4 *>(row + 64);
          a[0][j] = v0.x; a[1][j] = v0.y; a[2][j] = v0.z; a[3][j] = v0.w;
          a[4][j] = v1.x; a[5][j] = v1.y; a[6][j] = v1.z; a[7][j] = v1.w;
        }
      }
#pragma unroll
      for (int j = 0; j < KA; ++j) {
        const int kk = kg * KA + j;
        float b[TN];
        if (Cfg::B_KMAJOR) {
#pragma unroll
          for (int c = 0; c < TN; ++c) b[c] = bk[kk][c];
        } else {
          const char *row = b_base + (kc * 4 + kk) * BN * 4;
#pragma unroll
          for (int h = 0; h < TN / 4; ++h) {
            const float4 v = *reinterpret_cast<const float4 *>(row + h * 128);
            b[4 * h + 0] = v.x; b[4 * h + 1] = v.y; b[4 * h + 2] = v.z; b[4 * h + 3] = v.w;
          }
        }
        if (MODE == kPairCols) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float2 ar = make_float2(a[r][j], a[r][j]);
#pragma unroll
            for (int q = 0; q < TN / 2; ++q)
              acc[r * (TN / 2) + q] =
                  __ffma2_rn(ar, make_float2(b[2 * q], b[2 * q + 1]), acc[r * (TN / 2) + q]);
          }
        } else if (MODE == kPairRows) {
#pragma unroll
          for (int c = 0; c < TN; ++c) {
            const float2 bc = make_float2(b[c], b[c]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              acc[q * TN + c] = __ffma2_rn(make_float2(a[2 * q][j], a[2 * q + 1][j]), bc, acc[q * TN + c]);
          }
        } else {
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < TN; ++c)
              acc_ref<kScalar, TN>(acc, r, c) = fmaf(a[r][j], b[c], acc_ref<kScalar, TN>(acc, r, c));
        }
      }
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void epilogue(const SimtParams &p, float *Cb, const AccT<Cfg> &acc,
                                         int m0, int n0, int wm, int wn, int tm, int tn) {
  constexpr int MODE = acc_mode<Cfg>(), TN = Cfg::TN;
  const bool read_c = p.beta != 0.0f;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int m = m0 + wm * 32 + thread_row<Cfg>(tm, r);
    if (m >= p.M || !SG_CHECK(m - m0 < Cfg::BM, p.status)) continue;
    float *crow = Cb + static_cast<int64_t>(m) * p.ldc;
    if (!Cfg::B_KMAJOR) {
      // columns 32h + 4tn .. +3: TN/4 float4 groups
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const int n = n0 + wn * Cfg::WN + h * 32 + 4 * tn;
        if (!SG_CHECK(n - n0 + 3 < Cfg::BN, p.status)) continue;
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = acc_get<MODE, TN>(acc, r, 4 * h + q);
        if (p.c_vec4 && n + 3 < p.N) {
          float4 o;
          if (read_c) {
            const float4 c = *reinterpret_cast<const float4 *>(crow + n);
            o.x = fmaf(p.alpha, v[0], p.beta * c.x);
            o.y = fmaf(p.alpha, v[1], p.beta * c.y);
            o.z = fmaf(p.alpha, v[2], p.beta * c.z);
            o.w = fmaf(p.alpha, v[3], p.beta * c.w);
          } else {
            o.x = p.alpha * v[0];
            o.y = p.alpha * v[1];
            o.z = p.alpha * v[2];
            o.w = p.alpha * v[3];
          }
          *reinterpret_cast<float4 *>(crow + n) = o;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (n + q < p.N)
              crow[n + q] = read_c ? fmaf(p.alpha, v[q], p.beta * crow[n + q]) : p.alpha * v[q];
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < TN; ++c) {
        const int n = n0 + wn * Cfg::WN + thread_col<Cfg>(tn, c);
        if (n < p.N && SG_CHECK(n - n0 < Cfg::BN, p.status)) {
          const float a = acc_get<MODE, TN>(acc, r, c);
          crow[n] = read_c ? fmaf(p.alpha, a, p.beta * crow[n]) : p.alpha * a;
        }
      }
    }
  }
}

// Raw sums of a k-segment (no alpha/beta) to a dense BM x BN workspace tile.
template <class Cfg>
__device__ __forceinline__ void store_partial(float *ws, const AccT<Cfg> &acc, int wm, int wn,
                                              int tm, int tn) {
  constexpr int MODE = acc_mode<Cfg>(), TN = Cfg::TN;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float *row = ws + static_cast<int64_t>(wm * 32 + thread_row<Cfg>(tm, r)) * Cfg::BN + wn * Cfg::WN;
    if (!Cfg::B_KMAJOR) {
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        float4 o;
        o.x = acc_get<MODE, TN>(acc, r, 4 * h + 0);
        o.y = acc_get<MODE, TN>(acc, r, 4 * h + 1);
        o.z = acc_get<MODE, TN>(acc, r, 4 * h + 2);
        o.w = acc_get<MODE, TN>(acc, r, 4 * h + 3);
        *reinterpret_cast<float4 *>(row + h * 32 + 4 * tn) = o;
      }
    } else {
#pragma unroll
      for (int c = 0; c < TN; ++c) row[thread_col<Cfg>(tn, c)] = acc_get<MODE, TN>(acc, r, c);
    }
  }
}

// 3-D TMA store (batch coordinate c2).
__device__ __forceinline__ void tma_store_3d(const void *desc, uint32_t src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(desc)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// alpha * acc into the staging tile: column block j = column / 32 holds rows
// of 128 bytes, 16-byte chunk q of row R at chunk q ^ (R mod 8) (the layout
// of a 128-byte-swizzled TMA box, 1024-byte aligned).
template <class Cfg>
__device__ __forceinline__ void stage_tile(unsigned char *staging, const AccT<Cfg> &acc, float alpha,
                                           int wm, int wn, int tm, int tn, int *status) {
  constexpr int MODE = acc_mode<Cfg>(), TN = Cfg::TN;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int R = wm * 32 + thread_row<Cfg>(tm, r);
    if (!Cfg::B_KMAJOR) {
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const int col = wn * Cfg::WN + h * 32 + 4 * tn;
        float4 o;
        o.x = alpha * acc_get<MODE, TN>(acc, r, 4 * h + 0);
        o.y = alpha * acc_get<MODE, TN>(acc, r, 4 * h + 1);
        o.z = alpha * acc_get<MODE, TN>(acc, r, 4 * h + 2);
        o.w = alpha * acc_get<MODE, TN>(acc, r, 4 * h + 3);
        unsigned char *dst = staging + (col >> 5) * (Cfg::BM * 128) + R * 128 +
                             ((((col & 31) >> 2) ^ (R & 7)) << 4);
        if (!SG_CHECK(R < Cfg::BM && col + 3 < Cfg::BN, status)) continue;
        *reinterpret_cast<float4 *>(dst) = o;
      }
    } else {
#pragma unroll
      for (int c = 0; c < TN; ++c) {
        const int col = wn * Cfg::WN + thread_col<Cfg>(tn, c);
        unsigned char *dst = staging + (col >> 5) * (Cfg::BM * 128) + R * 128 +
                             ((((col & 31) >> 2) ^ (R & 7)) << 4) + ((col & 3) << 2);
        *reinterpret_cast<float *>(dst) = alpha * acc_get<MODE, TN>(acc, r, c);
      }
    }
  }
}

// Kernels that can finish split tiles themselves (SimtParams::sk_count).
// SG_SK_INKERNEL_ATRANS 1: also the kernels whose producer warps transpose A.
#ifndef SG_SK_INKERNEL_ATRANS
#define SG_SK_INKERNEL_ATRANS 0
#endif
template <class Cfg>
__host__ __device__ constexpr bool kInKernelFixup() {
  return Cfg::PRODUCER == kTma && (!Cfg::A_TRANS || SG_SK_INKERNEL_ATRANS) && Cfg::MATH_WARPS == 8;
}

// Barrier of the math warps only (the producer warps never take part), on an
// mbarrier with one arrival per math warp, so that its wait is bounded like
// every other wait of the kernel; false if it gave up.
__device__ __forceinline__ bool math_barrier(uint32_t bar, uint32_t &phase, int lane, const SimtParams &p) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = wait_parity_bounded(bar, phase, p.wait_budget_ns, p.status);
  phase ^= 1u;
  return ok;
}

// acc += a partial tile stored by store_partial (read through L2: other CTAs
// wrote it during this launch).
template <class Cfg>
__device__ __forceinline__ void add_partial(AccT<Cfg> &acc, const float *ws, int wm, int wn, int tm,
                                            int tn) {
  constexpr int MODE = acc_mode<Cfg>(), TN = Cfg::TN;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float *row = ws + static_cast<int64_t>(wm * 32 + thread_row<Cfg>(tm, r)) * Cfg::BN + wn * Cfg::WN;
    if (!Cfg::B_KMAJOR) {
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(row + h * 32 + 4 * tn));
        acc_ref<MODE, TN>(acc, r, 4 * h + 0) += v.x;
        acc_ref<MODE, TN>(acc, r, 4 * h + 1) += v.y;
        acc_ref<MODE, TN>(acc, r, 4 * h + 2) += v.z;
        acc_ref<MODE, TN>(acc, r, 4 * h + 3) += v.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < TN; ++c) acc_ref<MODE, TN>(acc, r, c) += __ldcg(row + thread_col<Cfg>(tn, c));
    }
  }
}

// Cluster split-K reduction, once every CTA of the cluster has staged its
// partial (dense BM x BN at stg in each CTA's shared memory): the math threads
// of CTA `rank` add rows [rank*BM/S, (rank+1)*BM/S) of the S partials in rank
// order (0 + p0 + p1 + ...) through distributed shared memory, apply alpha
// and beta and write C.  Not inlined, and called after the unit loop: inlined
// (in the loop or after it) it raised the k-loop's register pressure.  The
// parameters are passed by value: through a reference to the kernel's
// parameters its loop ran about a third slower (1024^3 under a scratch limit
// of 0, clusters of two: 3.9 -> 3.1 us for a CTA's half tile).
template <class Cfg>
__device__ __noinline__ void csk_reduce(const SimtParams p, int tile, int S, uint32_t rank, uint32_t stg,
                                        int tid) {
  int bi, tile_m, tile_n;
  unit_coords(p, tile, bi, tile_m, tile_n);
  float *Cb = p.C + static_cast<int64_t>(bi) * p.strideC;
  const bool read_c = p.beta != 0.0f;
  constexpr int BN4 = Cfg::BN / 4;
  const int rows = Cfg::BM / S, r0 = static_cast<int>(rank) * rows;
  for (int e = tid; e < rows * BN4; e += Cfg::MATH_THREADS) {
    const int row = r0 + e / BN4, c4 = e % BN4;
    const int m = tile_m * Cfg::BM + row, n = tile_n * Cfg::BN + 4 * c4;
    if (m >= p.M || n >= p.N) continue;
    const uint32_t off = static_cast<uint32_t>(row * Cfg::BN + 4 * c4) * 4u;
    if (!SG_CHECK(row < Cfg::BM && rank < static_cast<uint32_t>(S) &&
                      off + 16 <= static_cast<uint32_t>(Cfg::BM * Cfg::BN * 4), p.status))
      continue;
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int q = 0; q < S; ++q) {
      const float4 v = ld_dsmem_v4(map_to_rank(stg + off, q));
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    float *crow = Cb + static_cast<int64_t>(m) * p.ldc;
    const float v[4] = {sum.x, sum.y, sum.z, sum.w};
    if (p.c_vec4 && n + 3 < p.N) {
      float4 o;
      if (read_c) {
        const float4 c = *reinterpret_cast<const float4 *>(crow + n);
        o = make_float4(fmaf(p.alpha, v[0], p.beta * c.x), fmaf(p.alpha, v[1], p.beta * c.y),
                        fmaf(p.alpha, v[2], p.beta * c.z), fmaf(p.alpha, v[3], p.beta * c.w));
      } else {
        o = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
      }
      *reinterpret_cast<float4 *>(crow + n) = o;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (n + q < p.N) crow[n + q] = read_c ? fmaf(p.alpha, v[q], p.beta * crow[n + q]) : p.alpha * v[q];
    }
  }
}

// ------------------------------------------------------------------ kernel
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_CTAS)
    simt_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const SimtParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_last;   // in-kernel fixup: this CTA arrived last at its tile
  __shared__ __align__(8) uint64_t s_math_bar;
  // cluster split-K: every partial of the cluster staged / every peer done reading
  __shared__ __align__(8) uint64_t s_csk_bar[2];
  // 1024-byte alignment of the stage ring (required by the 128 B swizzle).
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t full0 = smem_base + Cfg::BAR_OFFSET;
  const uint32_t empty0 = full0 + 8 * Cfg::STAGES;
  const uint32_t raw_full0 = empty0 + 8 * Cfg::STAGES;
  const uint32_t raw_empty0 = raw_full0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(full0 + 8 * s, Cfg::FULL_COUNT);
      mbar_init(empty0 + 8 * s, Cfg::MATH_WARPS);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(raw_full0 + 8 * r, 1);
      mbar_init(raw_empty0 + 8 * r, Cfg::TRANSPOSER_WARPS);
    }
    if constexpr (kInKernelFixup<Cfg>() || Cfg::EPI_TMA || Cfg::CSK)
      mbar_init(smem_u32(&s_math_bar), Cfg::MATH_WARPS);
    if constexpr (Cfg::CSK) {
      // one arrival per math warp of each of the cluster's CTAs
      mbar_init(smem_u32(&s_csk_bar[0]), p.csk * Cfg::MATH_WARPS);
      mbar_init(smem_u32(&s_csk_bar[1]), p.csk * Cfg::MATH_WARPS);
    }
    fence_mbar_init();
  }
  if (Cfg::PRODUCER == kTma && threadIdx.x == Cfg::MATH_THREADS) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Cfg::EPI_TMA && p.c_tma) tma_prefetch_desc(&tmC);
  }
  __syncthreads();
  // the peers' barriers exist before any CTA of the cluster arrives on them
  if constexpr (Cfg::CSK) cluster_sync();
  // Everything above overlaps the previous kernel of the same call (the
  // transpose of an operand) when this one was launched as its dependent; the
  // operands and C are touched only after it has finished.  The fixup pass
  // that follows may be scheduled as soon as CTA slots free up.
  griddep_wait();
  griddep_launch_dependents();

  bool ok = true;
  if (warp >= Cfg::MATH_WARPS) {
    // ---------------- producer role
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::PRODUCER_REGS));
    if (Cfg::PRODUCER == kTma) {
      if (threadIdx.x == Cfg::MATH_THREADS)
        produce_tma<Cfg>(p, &tmA, &tmB, &tmC, smem_base, full0, empty0, raw_full0, raw_empty0, ok);
      else if (Cfg::A_TRANS && warp > Cfg::MATH_WARPS && warp <= Cfg::MATH_WARPS + Cfg::TRANSPOSER_WARPS)
        transpose_a<Cfg>(p, smem, full0, empty0, raw_full0, raw_empty0, warp - Cfg::MATH_WARPS - 1,
                         lane, ok);
    } else {
      produce_cpasync<Cfg>(p, smem_base, full0, empty0, threadIdx.x - Cfg::MATH_THREADS, ok);
    }
    return;
  }

  // ---------------- math role
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::MATH_REGS));
  const int wm = warp / Cfg::WARPS_N;
  const int wn = warp % Cfg::WARPS_N;
  const int tm = lane >> 3;
  const int tn = lane & 7;
  uint32_t it = 0;
  const uint32_t math_bar = smem_u32(&s_math_bar);
  uint32_t math_phase = 0;
  // Writes a finished tile (alpha applied) to C: through the staging tile and
  // TMA stores when p.c_tma, else straight from registers.  False if a
  // bounded wait gave up.
  const auto finish_tile = [&](const AccT<Cfg> &acc, int tile) -> bool {
    // tile coordinates only now: nothing but acc stays live across the k-loop
    int bi, tile_m, tile_n;
    unit_coords(p, tile, bi, tile_m, tile_n);
    if constexpr (Cfg::EPI_TMA) {
      if (p.c_tma) {
        // the previous tile's stores have read the staging tile
        if (threadIdx.x == 0) bulk_wait_group_read<0>();
        if (!math_barrier(math_bar, math_phase, lane, p)) return false;
        stage_tile<Cfg>(smem + Cfg::STAGING_OFFSET, acc, p.alpha, wm, wn, tm, tn, p.status);
        fence_proxy_async_smem();
        if (!math_barrier(math_bar, math_phase, lane, p)) return false;
        if (threadIdx.x == 0) {
          const int m0 = tile_m * Cfg::BM, n0 = tile_n * Cfg::BN;
#pragma unroll
          for (int j = 0; j < Cfg::BN / 32; ++j) {
            if (n0 + 32 * j >= p.N) break;
            const uint32_t src = smem_base + Cfg::STAGING_OFFSET + j * (Cfg::BM * 128);
            if (p.c_tma == 2)
              tma_store_3d(&tmC, src, n0 + 32 * j, m0, bi);
            else
              tma_store_2d(&tmC, src, n0 + 32 * j, m0);
          }
          bulk_commit_group();
        }
        return true;
      }
    }
    epilogue<Cfg>(p, p.C + static_cast<int64_t>(bi) * p.strideC, acc, tile_m * Cfg::BM,
                  tile_n * Cfg::BN, wm, wn, tm, tn);
    return true;
  };
  // Cluster split-K, first half: stages this CTA's partial tile in its own
  // (now idle) stage ring and announces it to every CTA of the cluster.  The
  // second half -- the reduction -- runs after the unit loop, where nothing
  // of the k-loop is live.  False if a bounded wait gave up.
  int csk_tile = -1;
  const auto csk_stage = [&](const AccT<Cfg> &acc, int tile) -> bool {
    // every math warp is past its last stage: the ring may be overwritten
    if (!math_barrier(math_bar, math_phase, lane, p)) return false;
    store_partial<Cfg>(reinterpret_cast<float *>(smem), acc, wm, wn, tm, tn);
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
    __syncwarp();
    if (lane == 0)
      for (int q = 0; q < p.csk; ++q) mbar_arrive_cluster(map_to_rank(smem_u32(&s_csk_bar[0]), q));
    csk_tile = tile;
    return true;
  };
  for_each_unit<Cfg::CSK>(p, [&](const WorkUnit &u) {
    AccT<Cfg> acc;
#pragma unroll
    for (int q = 0; q < 4 * Cfg::TN; ++q) acc[q] = make_float2(0.0f, 0.0f);

    for (int kt = u.k0; kt < u.k1; ++kt, ++it) {
      const uint32_t s = it % Cfg::STAGES;
      const uint32_t round = it / Cfg::STAGES;
      if (!wait_parity_bounded(full0 + 8 * s, round & 1, p.wait_budget_ns, p.status)) return false;
      const char *a_stage = reinterpret_cast<const char *>(smem) + s * Cfg::STAGE_BYTES;
      mma_stage<Cfg>(acc, a_stage, a_stage + Cfg::A_STAGE_BYTES, wm, wn, tm, tn, p.status);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if constexpr (Cfg::CSK) return csk_stage(acc, u.tile);
    if constexpr (!kInKernelFixup<Cfg>()) {
      if (u.slot < 0) {
        return finish_tile(acc, u.tile);
      } else {
        // sk_fixup_kernel adds the partials (these kernels run the mid-size
        // products, for which the separate pass is the faster)
        if (SG_CHECK(u.slot < 2 * static_cast<int>(gridDim.x), p.status))
          store_partial<Cfg>(p.workspace + static_cast<int64_t>(u.slot) * Cfg::BM * Cfg::BN, acc, wm, wn,
                             tm, tn);
      }
      return true;
    }
    if (u.slot >= 0) {
      if (SG_CHECK(u.slot < 2 * static_cast<int>(gridDim.x), p.status))
        store_partial<Cfg>(p.workspace + static_cast<int64_t>(u.slot) * Cfg::BM * Cfg::BN, acc, wm, wn,
                           tm, tn);
      if (p.sk_count == nullptr) return true;   // sk_fixup_kernel adds the partials
      // count this segment in; the last to arrive adds the tile's partials
      const int ts = u.tile - p.dp_tiles;
      int own = -1;
      const int n = sk_for_each_segment(p, gridDim.x, ts, [&](int i, int slot) {
        if (slot == u.slot) own = i;
      });
      __threadfence();
      if (!math_barrier(math_bar, math_phase, lane, p)) return false;
      if (threadIdx.x == 0) {
        const bool last = atomicAdd(p.sk_count + ts, 1) == n - 1;
        if (last) p.sk_count[ts] = 0;   // ready for the next launch
        s_last = last;
        __threadfence();
      }
      if (!math_barrier(math_bar, math_phase, lane, p)) return false;
      if (!s_last) return true;
      // the sum in k order, 0 + p0 + p1 + ..., as sk_fixup_kernel forms it;
      // this CTA's own partial is still in acc when it comes first
      constexpr int MODE = acc_mode<Cfg>(), TN = Cfg::TN;
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < TN; ++c)
          acc_ref<MODE, TN>(acc, r, c) = own == 0 ? 0.0f + acc_get<MODE, TN>(acc, r, c) : 0.0f;
      sk_for_each_segment(p, gridDim.x, ts, [&](int i, int slot) {
        if (i == 0 && own == 0) return;
        if (!SG_CHECK(slot >= 0 && slot < 2 * static_cast<int>(gridDim.x), p.status)) return;
        add_partial<Cfg>(acc, p.workspace + static_cast<int64_t>(slot) * Cfg::BM * Cfg::BN, wm, wn, tm, tn);
      });
    }
    return finish_tile(acc, u.tile);
  });
  // Cluster split-K, second half: once every CTA of the cluster has staged
  // its partial, this CTA adds rows [rank*BM/S, (rank+1)*BM/S) of the S
  // partials in rank order (0 + p0 + p1 + ...) through distributed shared
  // memory, applies alpha / beta and writes C; then it keeps its shared
  // memory until every peer has read it.
  if constexpr (Cfg::CSK) {
    if (csk_tile < 0) return;   // a bounded wait gave up before the partial was staged
    const int S = p.csk;
    const uint32_t rank = blockIdx.x % static_cast<uint32_t>(S);
    const uint32_t full = smem_u32(&s_csk_bar[0]), done = smem_u32(&s_csk_bar[1]);
    if (!wait_parity_bounded_cluster(full, 0, p.wait_budget_ns, p.status)) return;
    csk_reduce<Cfg>(p, csk_tile, S, rank, smem_u32(smem), threadIdx.x);
    __syncwarp();
    if (lane == 0)
      for (int q = 0; q < S; ++q) mbar_arrive_cluster(map_to_rank(done, q));
    wait_parity_bounded_cluster(done, 0, p.wait_budget_ns, p.status);
    return;
  }
  // the last tile's TMA stores complete before the CTA (and its shared
  // memory) goes away
  if constexpr (Cfg::EPI_TMA) {
    if (threadIdx.x == 0 && p.c_tma) bulk_wait_group_all();
  }
}

}  // namespace sg
