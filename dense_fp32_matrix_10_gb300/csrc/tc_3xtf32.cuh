// tc_3xtf32.cuh -- FP32 GEMM on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators) with the 3xTF32 split.
//
// Every FP32 operand x is taken as the sum of two TF32 values,
//     x_big   = x with its low 13 mantissa bits dropped (what the tensor core
//               reads when handed the FP32 word itself),
//     x_small = tf32(x - x_big)   (x - x_big is exact in FP32; rounded to nearest),
// and each product as a_small*b_big + a_big*b_small + a_big*b_big: three
// kind::tf32 MMAs accumulating in FP32 in tensor memory.  The dropped
// a_small*b_small term and the rounding of the small parts are ~2^-20 relative
// to |a*b|, below the FP32 accumulation error of a long dot product;
// integer-valued inputs of at most 11 significant bits have small = 0, so
// integer products stay exact.  Non-finite inputs get small = 0.
//
// B is read K-major from shared memory (128-byte rows of 32 k, 128 B swizzle);
// A too when it is k-contiguous, while an m-contiguous A (the layout the
// dispatcher gives every large product) is converted straight into tensor
// memory and read from there (measured on GB300 at 4096^3 TN: converters
// 172 -> 189 TFLOP/s with the paired split below, 217 with A in TMEM).
// Roles (one persistent CTA of 16 warps per SM, 128 x 128 output tiles, k in
// slices of 32):
//   warp 0       TMA producer.  A k-contiguous operand (A stored M x K, B stored
//                N x K) lands straight in the MMA ring as a [128][32] box and
//                serves as its own big part.  An m/n-contiguous operand lands in
//                a 2-stage raw ring as a dense [32 k][128 mn] box;
//   warps 8..15  converters: for a k-contiguous operand write small = tf32(x -
//                x_big) beside the raw tile (elementwise, same layout); for an
//                m/n-contiguous one build both x_big and x_small tiles K-major
//                from the raw ring (a transpose through shared memory);
//   warp 1       allocates 256 TMEM columns (two 128-column accumulators; 512
//                with A's parts in TMEM too); one thread issues 3 MMAs
//                (128 x 128 x 8) per k8;
//   warps 4..7   epilogue (warp 4+q owns TMEM lanes 32q..32q+31 = tile rows).
// Accuracy: the tensor core's FP32 accumulator rounds toward zero on every MMA
// (measured: a 4096-long accumulation drifts to ~3e-5 relative, linearly in K).
// So TMEM accumulates only CHUNK_KTILES k-slices (256 k) at a time; the
// epilogue warps add each finished chunk into FP32 registers with
// round-to-nearest adds and write C after the last chunk.  The directed error
// stays at the size of one chunk's, independent of K.
// All waits are bounded; on give-up every role leaves its loop, in-flight
// copies and MMAs are drained (bounded) and TMEM is freed before the CTA ends.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"
#include "simt_gemm.cuh"  // tile_coords

#ifndef SG_TC_A_TMEM
#define SG_TC_A_TMEM 1
#endif
#ifndef SG_TC_RAW_STAGES
#define SG_TC_RAW_STAGES 2
#endif
#ifndef SG_TC_ATMEM_STAGES
#define SG_TC_ATMEM_STAGES 3
#endif
#ifndef SG_TC_ATMEM_RAW_STAGES
#define SG_TC_ATMEM_RAW_STAGES 3
#endif

namespace sg {

struct TcParams {
  float *C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int tiles_m, tiles_n, k_tiles, num_tiles;
  // CTA-pair kernel: work units [0, wide_tiles) are whole tiles; each unit
  // beyond is one column half of a later tile (two units per tile), so the
  // last, partial round of tiles is spread over twice the units
  int wide_tiles;
  int group_m;
  int c_vec4;
  uint64_t wait_budget_ns;
  int *status;
};

template <bool A_KMAJOR_, bool B_KMAJOR_, bool PRESPLIT_ = false, int BN_ = 128>
struct TcConfig {
  static constexpr bool A_KMAJOR = A_KMAJOR_;
  static constexpr bool B_KMAJOR = B_KMAJOR_;
  // PRESPLIT: the small parts come from global memory (written by a split
  // pass before the launch) and land in the stage by TMA like the big parts;
  // the converter warps have nothing to do.
  static constexpr bool PRESPLIT = PRESPLIT_;
  static_assert(!PRESPLIT || (A_KMAJOR && B_KMAJOR), "pre-split operands are K-major");
  // BN = 256 (pre-split form only): 128 x 256 tiles, one 128 x 256 x 8 MMA
  // per product term.  The MMAs read both operands from shared memory, and
  // at 128 x 128 that read (8 KiB per MMA) bounds them: a run without any
  // TMA refill was no more than 5 % faster.  The wide MMA reads 12 KiB for
  // twice the work.
  static constexpr int BM = 128, BN = BN_, BK = 32;
  static_assert(BN == 128 || (BN == 256 && PRESPLIT_), "256-wide tiles: pre-split form only");
  static constexpr int TILE_BYTES = 128 * 32 * 4;  // one 128 x 32 FP32 tile
  static constexpr int B_TILE_BYTES = BN * 32 * 4;
  // A_TMEM: an m-contiguous A (through the raw ring) is converted straight
  // into tensor memory and the MMAs read it from there, so shared memory
  // carries only B for them (its bandwidth bounds this kernel).
  static constexpr bool A_TMEM = !A_KMAJOR && SG_TC_A_TMEM;
  // MMA ring stage: A big, A small (unless A_TMEM), B big, B small (K-major,
  // 128 B swizzle).  A k-contiguous operand's big tile is its raw TMA tile.
  static constexpr int STAGE_BYTES = (A_TMEM ? 0 : 2 * TILE_BYTES) + 2 * B_TILE_BYTES;
  static constexpr int A_BIG = 0, A_SMALL = TILE_BYTES, B_BIG = A_TMEM ? 0 : 2 * TILE_BYTES,
                       B_SMALL = B_BIG + B_TILE_BYTES;
  // Raw ring: the m/n-contiguous operands' FP32 slices, dense [32 k][128 mn].
  static constexpr int RAW_OPERANDS = (A_KMAJOR ? 0 : 1) + (B_KMAJOR ? 0 : 1);
  // Raw-ring depth: a TMA load must land within RAW_STAGES k-slices of MMA
  // work; with A in TMEM the smaller MMA stages leave room for a deeper ring.
  static constexpr int RAW_STAGES = RAW_OPERANDS ? (A_TMEM ? SG_TC_ATMEM_RAW_STAGES : SG_TC_RAW_STAGES) : 0;
  static constexpr int RAW_STAGE_BYTES = RAW_OPERANDS * TILE_BYTES;
  // (BN = 256: two stages of 96 KiB)
  static constexpr int STAGES =
      A_TMEM ? SG_TC_ATMEM_STAGES : ((RAW_OPERANDS == 2 || BN == 256) ? 2 : 3);
  // TMEM columns: two BN-column accumulators, then (A_TMEM) per stage A big
  // (32 columns = 32 k) and A small (32 more).
  static constexpr int A_TMEM_COL = 256;
  static constexpr int TMEM_COLS = (A_TMEM || BN == 256) ? 512 : 256;
  static_assert(!A_TMEM || A_TMEM_COL + 64 * STAGES <= TMEM_COLS, "A stages exceed TMEM");
  static constexpr int RAW_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int RAW_A = 0, RAW_B = A_KMAJOR ? 0 : TILE_BYTES;  // within a raw stage
  static constexpr int BAR_OFFSET = RAW_OFFSET + RAW_STAGES * RAW_STAGE_BYTES;
  // full, conv_full, empty per stage; raw_full, raw_empty per raw stage;
  // acc_full[2], acc_empty[2]; drain
  static constexpr int RAW_BARS = RAW_STAGES > 0 ? RAW_STAGES : 1;
  static constexpr int NUM_BARS = 3 * STAGES + 2 * RAW_BARS + 4 + 1;
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
  // BN = 256: three warpgroups (no converters; the tile's two 128-column
  // halves go to two epilogue warpgroups)
  static constexpr int THREADS = BN == 256 ? 384 : 512;
  static constexpr uint32_t IDESC = idesc_tf32(128, BN);
  // Two converter warpgroups: the conversion is ~250 dependent instructions
  // per thread and k-slice with one warpgroup, more than the 768 tensor-core
  // cycles of the slice's 12 MMAs.
  static constexpr int CONVERTER_WARPS = 8;
  static constexpr int CONVERTER_THREADS = 32 * CONVERTER_WARPS;
  static constexpr int EPILOGUE_WARPS = BN / 32;
  static constexpr int CHUNK_KTILES = 8;  // k-slices accumulated in TMEM per promotion
  // setmaxnreg split by warpgroup: {producer, MMA, idle}, epilogue (holds a
  // 128-float half row of the tile), then two converter warpgroups or (BN =
  // 256) the second epilogue warpgroup.
  static constexpr int REGS_WG0 = BN == 256 ? 40 : 56, REGS_EPI = BN == 256 ? 232 : 240,
                       REGS_CONV = 104;
  static constexpr int REGS_SPLIT =
      128 * (REGS_WG0 + (BN == 256 ? 2 * REGS_EPI : REGS_EPI + 2 * REGS_CONV));
  static_assert(REGS_SPLIT <= THREADS * ((65536 / THREADS) & ~7),
                "register split exceeds the launch budget");
};

template <class Cfg>
struct TcBars {
  uint32_t base;
  __device__ uint32_t full(uint32_t s) const { return base + 8 * s; }
  __device__ uint32_t conv_full(uint32_t s) const { return base + 8 * (Cfg::STAGES + s); }
  __device__ uint32_t empty(uint32_t s) const { return base + 8 * (2 * Cfg::STAGES + s); }
  __device__ uint32_t raw_full(uint32_t r) const { return base + 8 * (3 * Cfg::STAGES + r); }
  __device__ uint32_t raw_empty(uint32_t r) const {
    return base + 8 * (3 * Cfg::STAGES + Cfg::RAW_BARS + r);
  }
  __device__ uint32_t acc_full(uint32_t b) const {
    return base + 8 * (3 * Cfg::STAGES + 2 * Cfg::RAW_BARS + b);
  }
  __device__ uint32_t acc_empty(uint32_t b) const {
    return base + 8 * (3 * Cfg::STAGES + 2 * Cfg::RAW_BARS + 2 + b);
  }
  __device__ uint32_t drain() const { return base + 8 * (3 * Cfg::STAGES + 2 * Cfg::RAW_BARS + 4); }
};

// ------------------------------------------------------------------ producer
template <class Cfg>
__device__ __forceinline__ void tc_produce(const TcParams &p, const CUtensorMap *tmA,
                                           const CUtensorMap *tmB, const CUtensorMap *tmAs,
                                           const CUtensorMap *tmBs, uint32_t sbase,
                                           const TcBars<Cfg> &bar) {
  constexpr bool ANY_K = Cfg::A_KMAJOR || Cfg::B_KMAJOR;
  constexpr uint32_t K_BYTES =
      Cfg::PRESPLIT ? Cfg::STAGE_BYTES
                    : ((Cfg::A_KMAJOR ? 1 : 0) + (Cfg::B_KMAJOR ? 1 : 0)) * Cfg::TILE_BYTES;
  uint32_t it = 0;        // k-slices whose copies are all issued
  bool k_issued = false;  // the k-contiguous part of slice `it` is issued
  bool ok = true;
  for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
    int tm, tn;
    tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * Cfg::BM, n0 = tn * Cfg::BN;
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it, k_issued = false) {
      const int k0 = kt * Cfg::BK;
      if (ANY_K) {  // k-contiguous operands straight into the MMA ring
        const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
        if (round > 0 &&
            !wait_parity_bounded(bar.empty(s), (round - 1) & 1, p.wait_budget_ns, p.status)) {
          ok = false;
          break;
        }
        const uint32_t st = sbase + s * Cfg::STAGE_BYTES;
        mbar_arrive_expect_tx(bar.full(s), K_BYTES);
        if (Cfg::A_KMAJOR) tma_load_2d(st + Cfg::A_BIG, tmA, bar.full(s), k0, m0);
        // op(B) in boxes of 128 n rows (two for a 256-wide tile, stacked)
#pragma unroll
        for (int h = 0; h < Cfg::BN / 128; ++h)
          if (Cfg::B_KMAJOR)
            tma_load_2d(st + Cfg::B_BIG + h * Cfg::TILE_BYTES, tmB, bar.full(s), k0, n0 + 128 * h);
        if (Cfg::PRESPLIT) {
          tma_load_2d(st + Cfg::A_SMALL, tmAs, bar.full(s), k0, m0);
#pragma unroll
          for (int h = 0; h < Cfg::BN / 128; ++h)
            tma_load_2d(st + Cfg::B_SMALL + h * Cfg::TILE_BYTES, tmBs, bar.full(s), k0, n0 + 128 * h);
        }
        k_issued = true;
      }
      if constexpr (Cfg::RAW_OPERANDS > 0) {  // m/n-contiguous operands into the raw ring
        const uint32_t r = it % Cfg::RAW_STAGES, rround = it / Cfg::RAW_STAGES;
        if (rround > 0 &&
            !wait_parity_bounded(bar.raw_empty(r), (rround - 1) & 1, p.wait_budget_ns, p.status)) {
          ok = false;
          break;
        }
        const uint32_t rs = sbase + Cfg::RAW_OFFSET + r * Cfg::RAW_STAGE_BYTES;
        mbar_arrive_expect_tx(bar.raw_full(r), Cfg::RAW_STAGE_BYTES);
        if (!Cfg::A_KMAJOR) tma_load_2d(rs + Cfg::RAW_A, tmA, bar.raw_full(r), m0, k0);
        if (!Cfg::B_KMAJOR) tma_load_2d(rs + Cfg::RAW_B, tmB, bar.raw_full(r), n0, k0);
      }
    }
  }
  if (!ok) {  // let issued copies land before the CTA can end (bounded waits)
    constexpr uint32_t DEPTH = Cfg::STAGES > Cfg::RAW_STAGES ? Cfg::STAGES : Cfg::RAW_STAGES;
    const uint32_t first = it > DEPTH ? it - DEPTH : 0;
    for (uint32_t j = first; j < it; ++j) {
      if (ANY_K)
        wait_parity_bounded(bar.full(j % Cfg::STAGES), (j / Cfg::STAGES) & 1, p.wait_budget_ns,
                            nullptr);
      if constexpr (Cfg::RAW_OPERANDS > 0)
        wait_parity_bounded(bar.raw_full(j % Cfg::RAW_STAGES), (j / Cfg::RAW_STAGES) & 1,
                            p.wait_budget_ns, nullptr);
    }
    if (k_issued)
      wait_parity_bounded(bar.full(it % Cfg::STAGES), (it / Cfg::STAGES) & 1, p.wait_budget_ns,
                          nullptr);
  }
}

// ------------------------------------------------------------------ converters
__device__ __forceinline__ float small_part(float x, float big) {
  return isfinite(x) ? to_tf32(x - big) : 0.0f;
}

#ifndef SG_TC_SPLIT_PAIR
#define SG_TC_SPLIT_PAIR 1
#endif

// k-contiguous operand: small = tf32(x - x_big) beside the raw tile, elementwise
// (same layout, so the small tile shares the raw tile's descriptor geometry).
// ct = converter thread 0..255; 1024 16-byte chunks, 4 per thread.
__device__ __forceinline__ void small_of_kmajor(const unsigned char *raw, unsigned char *small,
                                                int ct) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int off = (ct + 256 * i) * 16;
    const float4 x = *reinterpret_cast<const float4 *>(raw + off);
    float4 s;
    if (SG_TC_SPLIT_PAIR) {
      float b0, b1, b2, b3;
      split_pair(x.x, x.y, b0, b1, s.x, s.y);
      split_pair(x.z, x.w, b2, b3, s.z, s.w);
    } else {
      s.x = small_part(x.x, tf32_trunc(x.x));
      s.y = small_part(x.y, tf32_trunc(x.y));
      s.z = small_part(x.z, tf32_trunc(x.z));
      s.w = small_part(x.w, tf32_trunc(x.w));
    }
    *reinterpret_cast<float4 *>(small + off) = s;
  }
}

// m/n-contiguous operand: raw [32 k][128 mn] -> K-major big and small tiles
// (128-byte rows of 32 k, 128 B swizzle); converter thread ct builds half of
// row ct % 128 (k chunks 4*(ct / 128) .. +3).
__device__ __forceinline__ void split_of_mnmajor(const unsigned char *raw, unsigned char *big,
                                                 unsigned char *small, int ct0) {
  const float *r = reinterpret_cast<const float *>(raw);
  const int ct = ct0 & 127, half = ct0 >> 7;
#pragma unroll
  for (int kq = 0; kq < 4; ++kq) {
    const int kc = 4 * half + kq;
    float4 x;
    x.x = r[(4 * kc + 0) * 128 + ct];
    x.y = r[(4 * kc + 1) * 128 + ct];
    x.z = r[(4 * kc + 2) * 128 + ct];
    x.w = r[(4 * kc + 3) * 128 + ct];
    float4 b, s;
    if (SG_TC_SPLIT_PAIR) {
      split_pair(x.x, x.y, b.x, b.y, s.x, s.y);
      split_pair(x.z, x.w, b.z, b.w, s.z, s.w);
    } else {
      b.x = tf32_trunc(x.x);
      b.y = tf32_trunc(x.y);
      b.z = tf32_trunc(x.z);
      b.w = tf32_trunc(x.w);
      s.x = small_part(x.x, b.x);
      s.y = small_part(x.y, b.y);
      s.z = small_part(x.z, b.z);
      s.w = small_part(x.w, b.w);
    }
    const int off = ct * 128 + ((kc ^ (ct & 7)) << 4);
    *reinterpret_cast<float4 *>(big + off) = b;
    *reinterpret_cast<float4 *>(small + off) = s;
  }
}

// m-contiguous A slice, raw [32 k][128 m] -> TF32 big and small parts in
// tensor memory (A_TMEM): thread ct handles tile row m = ct % 128, which is
// lane l of its warp in TMEM lane quarter warp % 4 (m = 32 * (warp % 4) + l);
// the two converter warpgroups take k 0..15 and 16..31.
template <class Cfg>
__device__ __forceinline__ void a_to_tmem(const unsigned char *raw, uint32_t a_col, int ct, int warp) {
  const float *r = reinterpret_cast<const float *>(raw);
  const int m = ct & 127, kh = ct >> 7;
  uint32_t big[16], small[16];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float x0 = r[(16 * kh + j) * 128 + m], x1 = r[(16 * kh + j + 1) * 128 + m];
    float b0, b1, s0, s1;
    split_pair(x0, x1, b0, b1, s0, s1);
    big[j] = __float_as_uint(b0);
    big[j + 1] = __float_as_uint(b1);
    small[j] = __float_as_uint(s0);
    small[j + 1] = __float_as_uint(s1);
  }
  const uint32_t lanes = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  tmem_st_32x32b_x16(a_col + lanes + 16 * kh, big);
  tmem_st_32x32b_x16(a_col + lanes + 32 + 16 * kh, small);
  tmem_st_wait();
}

template <class Cfg>
__device__ __forceinline__ void tc_convert(const TcParams &p, unsigned char *smem,
                                           const TcBars<Cfg> &bar, uint32_t tmem_base, int ct,
                                           int warp, int lane) {
  constexpr bool ANY_K = Cfg::A_KMAJOR || Cfg::B_KMAJOR;
  if (Cfg::PRESPLIT) return;   // the split pass did their work
  uint32_t it = 0;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
      const uint32_t s = it % Cfg::STAGES, round = it / Cfg::STAGES;
      const uint32_t r = Cfg::RAW_OPERANDS ? it % Cfg::RAW_STAGES : 0;
      const uint32_t rround = Cfg::RAW_OPERANDS ? it / Cfg::RAW_STAGES : 0;
      // The stage is free once the MMAs of its previous round finished.  With
      // a k-contiguous operand the producer waited for that before its copy,
      // so the stage's `full` phase already implies it.
      if (!ANY_K && round > 0 &&
          !wait_parity_bounded(bar.empty(s), (round - 1) & 1, p.wait_budget_ns, p.status))
        return;
      if (ANY_K && !wait_parity_bounded(bar.full(s), round & 1, p.wait_budget_ns, p.status)) return;
      if (Cfg::RAW_OPERANDS &&
          !wait_parity_bounded(bar.raw_full(r), rround & 1, p.wait_budget_ns, p.status))
        return;
      unsigned char *st = smem + s * Cfg::STAGE_BYTES;
      const unsigned char *rs = smem + Cfg::RAW_OFFSET + r * Cfg::RAW_STAGE_BYTES;
      if (Cfg::A_TMEM) {
        tc_fence_after_sync();   // the MMAs that read this A stage have finished
        a_to_tmem<Cfg>(rs + Cfg::RAW_A, tmem_base + Cfg::A_TMEM_COL + 64 * s, ct, warp);
      } else if (Cfg::A_KMAJOR) {
        small_of_kmajor(st + Cfg::A_BIG, st + Cfg::A_SMALL, ct);
      } else {
        split_of_mnmajor(rs + Cfg::RAW_A, st + Cfg::A_BIG, st + Cfg::A_SMALL, ct);
      }
      if (Cfg::B_KMAJOR)
        small_of_kmajor(st + Cfg::B_BIG, st + Cfg::B_SMALL, ct);
      else
        split_of_mnmajor(rs + Cfg::RAW_B, st + Cfg::B_BIG, st + Cfg::B_SMALL, ct);
      fence_proxy_async_smem();  // the MMA reads these through the async proxy
      if (Cfg::A_TMEM) tc_fence_before_sync();   // ... and A's tensor-memory parts
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar.conv_full(s));
        if (Cfg::RAW_OPERANDS) mbar_arrive(bar.raw_empty(r));
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issue
template <class Cfg>
__device__ __forceinline__ void tc_issue(const TcParams &p, uint32_t sbase, uint32_t tmem_base,
                                         const TcBars<Cfg> &bar) {
  uint32_t it = 0, chunk_iter = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
    for (int kc0 = 0; kc0 < p.k_tiles && ok; kc0 += Cfg::CHUNK_KTILES, ++chunk_iter) {
      const uint32_t b = chunk_iter & 1, use = chunk_iter >> 1;
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
        if (!wait_parity_bounded(Cfg::PRESPLIT ? bar.full(s) : bar.conv_full(s), round & 1,
                                 p.wait_budget_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t st = sbase + s * Cfg::STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < Cfg::BK / 8; ++kk) {
          // k8 step kk: 32 bytes along the 128-byte K-major rows (8 TMEM columns)
          const uint64_t b_big = desc_kmajor_sw128(st + Cfg::B_BIG + kk * 32);
          const uint64_t b_small = desc_kmajor_sw128(st + Cfg::B_SMALL + kk * 32);
          const uint32_t acc = (kt > kc0 || kk > 0) ? 1u : 0u;
          if (Cfg::A_TMEM) {
            const uint32_t a_big = tmem_base + Cfg::A_TMEM_COL + 64 * s + 8 * kk;
            mma_tf32_a_tmem(d, a_big + 32, b_big, Cfg::IDESC, acc);   // a_small * b_big
            mma_tf32_a_tmem(d, a_big, b_small, Cfg::IDESC, 1u);
            mma_tf32_a_tmem(d, a_big, b_big, Cfg::IDESC, 1u);
          } else {
            const uint64_t a_big = desc_kmajor_sw128(st + Cfg::A_BIG + kk * 32);
            const uint64_t a_small = desc_kmajor_sw128(st + Cfg::A_SMALL + kk * 32);
            mma_tf32(d, a_small, b_big, Cfg::IDESC, acc);
            mma_tf32(d, a_big, b_small, Cfg::IDESC, 1u);
            mma_tf32(d, a_big, b_big, Cfg::IDESC, 1u);
          }
        }
        mma_commit(bar.empty(s));  // frees the stage when these MMAs finish
      }
      if (!ok) break;
      mma_commit(bar.acc_full(b));  // chunk done: hand the accumulator to the epilogue
    }
  }
  // Every MMA this thread issued must be complete before TMEM is freed.
  mma_commit(bar.drain());
  wait_parity_bounded(bar.drain(), 0, p.wait_budget_ns, nullptr);
}

// ------------------------------------------------------------------ epilogue
// C[row][n0 .. n0+127] = alpha * acc + beta * C (C not read when beta = 0);
// float4 where C allows it, elementwise at the ragged right edge.
__device__ __forceinline__ void tc_store_row(const TcParams &p, int row, int n0,
                                             const float (&acc)[128]) {
  if (row >= p.M) return;
  const bool read_c = p.beta != 0.0f;
  float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
  for (int j = 0; j < 128; j += 4) {
    const int n = n0 + j;
    if (p.c_vec4 && n + 3 < p.N) {
      float4 o;
      if (read_c) {
        const float4 c = *reinterpret_cast<const float4 *>(crow + n);
        o.x = fmaf(p.alpha, acc[j + 0], p.beta * c.x);
        o.y = fmaf(p.alpha, acc[j + 1], p.beta * c.y);
        o.z = fmaf(p.alpha, acc[j + 2], p.beta * c.z);
        o.w = fmaf(p.alpha, acc[j + 3], p.beta * c.w);
      } else {
        o.x = p.alpha * acc[j + 0];
        o.y = p.alpha * acc[j + 1];
        o.z = p.alpha * acc[j + 2];
        o.w = p.alpha * acc[j + 3];
      }
      *reinterpret_cast<float4 *>(crow + n) = o;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (n + e < p.N)
          crow[n + e] = read_c ? fmaf(p.alpha, acc[j + e], p.beta * crow[n + e]) : p.alpha * acc[j + e];
    }
  }
}

// Warp q of epilogue warpgroup `half` owns tile rows 32q .. 32q+31 (TMEM
// lanes) and columns 128 * half .. +127.
template <class Cfg>
__device__ __forceinline__ void tc_epilogue(const TcParams &p, uint32_t tmem_base,
                                            const TcBars<Cfg> &bar, int q, int half, int lane) {
  constexpr int W = 128;   // columns per thread
  uint32_t chunk_iter = 0;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    float acc[W];  // this thread's half row of the tile, FP32 round-to-nearest sums
#pragma unroll
    for (int j = 0; j < W; ++j) acc[j] = 0.0f;
    for (int kc0 = 0; kc0 < p.k_tiles; kc0 += Cfg::CHUNK_KTILES, ++chunk_iter) {
      const uint32_t b = chunk_iter & 1, use = chunk_iter >> 1;
      if (!wait_parity_bounded(bar.acc_full(b), use & 1, p.wait_budget_ns, p.status)) return;
      tc_fence_after_sync();
#pragma unroll
      for (int cc = 0; cc < W / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + b * Cfg::BN + half * W + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(v[j]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.acc_empty(b));
    }
    int tm, tn;
    tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    tc_store_row(p, tm * Cfg::BM + 32 * q + lane, tn * Cfg::BN + half * W, acc);
  }
}

// ------------------------------------------------------------------ kernel
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc3_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmBs,
                    const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const TcBars<Cfg> bar{sbase + Cfg::BAR_OFFSET};
  const uint32_t tmem_slot = sbase + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(bar.full(s), 1);
      mbar_init(bar.conv_full(s), Cfg::CONVERTER_WARPS);
      mbar_init(bar.empty(s), 1);
    }
    for (int r = 0; r < Cfg::RAW_BARS; ++r) {
      mbar_init(bar.raw_full(r), 1);
      mbar_init(bar.raw_empty(r), Cfg::CONVERTER_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.acc_full(b), 1);
      mbar_init(bar.acc_empty(b), Cfg::EPILOGUE_WARPS);
    }
    mbar_init(bar.drain(), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Cfg::PRESPLIT) {
      tma_prefetch_desc(&tmAs);
      tma_prefetch_desc(&tmBs);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base =
      *reinterpret_cast<volatile uint32_t *>(smem + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8);
  // launched as the dependent of an operand transpose: set-up above overlaps
  // it, operands and C are touched only after it has finished
  griddep_wait();

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_WG0));
    if (warp == 0) {
      if (lane == 0) tc_produce<Cfg>(p, &tmA, &tmB, &tmAs, &tmBs, sbase, bar);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) tc_issue<Cfg>(p, sbase, tmem_base, bar);
      __syncwarp();
    }
  } else if (warp < 8 || Cfg::BN == 256) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_EPI));
    tc_epilogue<Cfg>(p, tmem_base, bar, warp & 3, (warp >> 2) - 1, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_CONV));
    tc_convert<Cfg>(p, smem, bar, tmem_base, threadIdx.x - 256, warp, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace sg
