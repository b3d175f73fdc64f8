// tc_3xtf32.cuh -- FP32 GEMM on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators) with the 3xTF32 split.
//
// Every FP32 operand x is split into two TF32 values,
//     x_big = tf32(x)            (round to nearest, 10 explicit mantissa bits)
//     x_small = tf32(x - x_big)  (x - x_big is exact in FP32)
// and each product is taken as a_small*b_big + a_big*b_small + a_big*b_big,
// three kind::tf32 MMAs accumulating in FP32 in tensor memory.  The dropped
// a_small*b_small term and the rounding of the small parts are ~2^-21 relative
// to |a*b|, below the FP32 accumulation error of a long dot product, so the
// result meets the same tolerance as the CUDA-core kernels; integers of at most
// 11 significant bits split exactly (small part 0), so integer-valued products
// stay exact.
//
// Roles (one persistent CTA of 12 warps per SM, 128 x 128 output tiles, k in
// slices of 32):
//   warp 0       TMA producer: FP32 op(A), op(B) k-slices into a 2-stage raw ring
//                (k-contiguous operands with the 128 B swizzle, m/n-contiguous
//                ones dense);
//   warps 8..11  converters: raw FP32 -> big and small TF32 tiles in the
//                K-major 128 B-swizzled layout the MMA reads (transposing the
//                m/n-contiguous operands on the way), 2-stage ring;
//   warp 1       allocates 256 TMEM columns (two 128-column accumulators) and
//                one thread issues 3 x 4 MMAs (128 x 128 x 8) per k-slice,
//                committing each slice to its ring barrier and each finished
//                tile to the epilogue;
//   warps 4..7   epilogue: tcgen05.ld of the accumulator (warp 4+q owns TMEM
//                lanes 32q..32q+31 = tile rows), alpha/beta, stores to C;
//                the other accumulator is being filled meanwhile.
// Accuracy: the tensor core's FP32 accumulator rounds toward zero on every MMA
// (measured: the error of a 4096-long accumulation grows to ~3e-5 relative,
// linearly in K).  So TMEM accumulates only CHUNK_KTILES k-slices (256 k) at a
// time; the epilogue warps add each finished chunk into FP32 registers with
// round-to-nearest adds, and write C after the last chunk.  The directed
// error then stays at the size of one chunk's, independent of K.
// All waits are bounded; on give-up every role leaves its loop, in-flight
// copies and MMAs are drained (bounded) and TMEM is freed before the CTA ends.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"
#include "simt_gemm.cuh"  // tile_coords

namespace sg {

struct TcParams {
  float *C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int tiles_m, tiles_n, k_tiles, num_tiles;
  int group_m;
  int c_vec4;
  uint64_t wait_budget_ns;
  int *status;
};

template <bool A_KMAJOR_, bool B_KMAJOR_>
struct TcConfig {
  static constexpr bool A_KMAJOR = A_KMAJOR_;
  static constexpr bool B_KMAJOR = B_KMAJOR_;
  static constexpr int BM = 128, BN = 128, BK = 32;
  static constexpr int RAW_STAGES = 2, CONV_STAGES = 2;
  static constexpr int TILE_BYTES = 128 * 32 * 4;          // one 128 x 32 FP32 tile
  static constexpr int RAW_STAGE_BYTES = 2 * TILE_BYTES;   // A, B
  static constexpr int CONV_STAGE_BYTES = 4 * TILE_BYTES;  // A big, A small, B big, B small
  static constexpr int RAW_OFFSET = 0;
  static constexpr int CONV_OFFSET = RAW_STAGES * RAW_STAGE_BYTES;
  static constexpr int BAR_OFFSET = CONV_OFFSET + CONV_STAGES * CONV_STAGE_BYTES;
  // raw_full, raw_empty, conv_full, conv_empty, acc_full[2], acc_empty[2], drain
  static constexpr int NUM_BARS = 2 * RAW_STAGES + 2 * CONV_STAGES + 4 + 1;
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr int TMEM_COLS = 256;
  static constexpr uint32_t IDESC = idesc_tf32(128, 128);
  static constexpr int CONVERTER_WARPS = 4;
  static constexpr int EPILOGUE_WARPS = 4;
  static constexpr int CHUNK_KTILES = 8;  // k-slices accumulated in TMEM per promotion
  // setmaxnreg split by warpgroup: {producer, MMA, idle}, epilogue (holds a
  // 128-float row of the tile), converters.
  static constexpr int REGS_WG0 = 56, REGS_EPI = 240, REGS_CONV = 200;
  static_assert(128 * (REGS_WG0 + REGS_EPI + REGS_CONV) <= THREADS * ((65536 / THREADS) & ~7),
                "register split exceeds the launch budget");
};

template <class Cfg>
struct TcBars {
  uint32_t base;
  __device__ uint32_t raw_full(uint32_t s) const { return base + 8 * s; }
  __device__ uint32_t raw_empty(uint32_t s) const { return base + 8 * (Cfg::RAW_STAGES + s); }
  __device__ uint32_t conv_full(uint32_t s) const { return base + 8 * (2 * Cfg::RAW_STAGES + s); }
  __device__ uint32_t conv_empty(uint32_t s) const {
    return base + 8 * (2 * Cfg::RAW_STAGES + Cfg::CONV_STAGES + s);
  }
  __device__ uint32_t acc_full(uint32_t b) const {
    return base + 8 * (2 * Cfg::RAW_STAGES + 2 * Cfg::CONV_STAGES + b);
  }
  __device__ uint32_t acc_empty(uint32_t b) const {
    return base + 8 * (2 * Cfg::RAW_STAGES + 2 * Cfg::CONV_STAGES + 2 + b);
  }
  __device__ uint32_t drain() const { return base + 8 * (2 * Cfg::RAW_STAGES + 2 * Cfg::CONV_STAGES + 4); }
};

// ------------------------------------------------------------------ producer
template <class Cfg>
__device__ __forceinline__ void tc_produce(const TcParams &p, const CUtensorMap *tmA,
                                           const CUtensorMap *tmB, uint32_t sbase,
                                           const TcBars<Cfg> &bar) {
  uint32_t it = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
    int tm, tn;
    tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * Cfg::BM, n0 = tn * Cfg::BN;
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
      const uint32_t s = it % Cfg::RAW_STAGES, round = it / Cfg::RAW_STAGES;
      if (round > 0 &&
          !wait_parity_bounded(bar.raw_empty(s), (round - 1) & 1, p.wait_budget_ns, p.status)) {
        ok = false;
        break;
      }
      const uint32_t a_dst = sbase + Cfg::RAW_OFFSET + s * Cfg::RAW_STAGE_BYTES;
      const uint32_t b_dst = a_dst + Cfg::TILE_BYTES;
      mbar_arrive_expect_tx(bar.raw_full(s), Cfg::RAW_STAGE_BYTES);
      const int k0 = kt * Cfg::BK;
      if (Cfg::A_KMAJOR)
        tma_load_2d(a_dst, tmA, bar.raw_full(s), k0, m0);
      else
        tma_load_2d(a_dst, tmA, bar.raw_full(s), m0, k0);
      if (Cfg::B_KMAJOR)
        tma_load_2d(b_dst, tmB, bar.raw_full(s), k0, n0);
      else
        tma_load_2d(b_dst, tmB, bar.raw_full(s), n0, k0);
    }
  }
  if (!ok) {  // let issued copies land before the CTA can end
    const uint32_t first = it > Cfg::RAW_STAGES ? it - Cfg::RAW_STAGES : 0;
    for (uint32_t j = first; j < it; ++j)
      wait_parity_bounded(bar.raw_full(j % Cfg::RAW_STAGES), (j / Cfg::RAW_STAGES) & 1,
                          p.wait_budget_ns, nullptr);
  }
}

// ------------------------------------------------------------------ converters
__device__ __forceinline__ void split4(const float4 x, float4 &big, float4 &small) {
  big.x = to_tf32(x.x);
  big.y = to_tf32(x.y);
  big.z = to_tf32(x.z);
  big.w = to_tf32(x.w);
  small.x = to_tf32(x.x - big.x);
  small.y = to_tf32(x.y - big.y);
  small.z = to_tf32(x.z - big.z);
  small.w = to_tf32(x.w - big.w);
}

// One 128 x 32 operand tile: raw FP32 (as the TMA left it) -> big and small
// TF32 tiles, K-major with the 128 B swizzle.  ct = converter thread 0..127.
template <bool KMAJOR>
__device__ __forceinline__ void convert_tile(const unsigned char *raw, unsigned char *big,
                                             unsigned char *small, int ct) {
  if (KMAJOR) {
    // Raw tile already has the destination layout: elementwise, chunk by chunk.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int off = (ct + 128 * i) * 16;
      const float4 x = *reinterpret_cast<const float4 *>(raw + off);
      float4 b, s;
      split4(x, b, s);
      *reinterpret_cast<float4 *>(big + off) = b;
      *reinterpret_cast<float4 *>(small + off) = s;
    }
  } else {
    // Raw tile is [32 k][128 mn] (512 B rows); thread ct builds row mn = ct.
    const float *r = reinterpret_cast<const float *>(raw);
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      float4 x;
      x.x = r[(4 * kc + 0) * 128 + ct];
      x.y = r[(4 * kc + 1) * 128 + ct];
      x.z = r[(4 * kc + 2) * 128 + ct];
      x.w = r[(4 * kc + 3) * 128 + ct];
      float4 b, s;
      split4(x, b, s);
      const int off = ct * 128 + ((kc ^ (ct & 7)) << 4);
      *reinterpret_cast<float4 *>(big + off) = b;
      *reinterpret_cast<float4 *>(small + off) = s;
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void tc_convert(const TcParams &p, unsigned char *smem,
                                           const TcBars<Cfg> &bar, int ct, int lane) {
  uint32_t it = 0;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
      const uint32_t rs = it % Cfg::RAW_STAGES, rr = it / Cfg::RAW_STAGES;
      const uint32_t cs = it % Cfg::CONV_STAGES, cr = it / Cfg::CONV_STAGES;
      if (!wait_parity_bounded(bar.raw_full(rs), rr & 1, p.wait_budget_ns, p.status)) return;
      if (cr > 0 &&
          !wait_parity_bounded(bar.conv_empty(cs), (cr - 1) & 1, p.wait_budget_ns, p.status))
        return;
      const unsigned char *raw_a = smem + Cfg::RAW_OFFSET + rs * Cfg::RAW_STAGE_BYTES;
      const unsigned char *raw_b = raw_a + Cfg::TILE_BYTES;
      unsigned char *cv = smem + Cfg::CONV_OFFSET + cs * Cfg::CONV_STAGE_BYTES;
      convert_tile<Cfg::A_KMAJOR>(raw_a, cv, cv + Cfg::TILE_BYTES, ct);
      convert_tile<Cfg::B_KMAJOR>(raw_b, cv + 2 * Cfg::TILE_BYTES, cv + 3 * Cfg::TILE_BYTES, ct);
      fence_proxy_async_smem();  // the MMA reads these through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar.raw_empty(rs));
        mbar_arrive(bar.conv_full(cs));
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
      const uint32_t d = tmem_base + b * 128;
      const int kc1 = min(kc0 + Cfg::CHUNK_KTILES, p.k_tiles);
      for (int kt = kc0; kt < kc1; ++kt, ++it) {
        const uint32_t cs = it % Cfg::CONV_STAGES, cr = it / Cfg::CONV_STAGES;
        if (!wait_parity_bounded(bar.conv_full(cs), cr & 1, p.wait_budget_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t cv = sbase + Cfg::CONV_OFFSET + cs * Cfg::CONV_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < Cfg::BK / 8; ++kk) {
          const uint64_t a_big = desc_kmajor_sw128(cv + kk * 32);
          const uint64_t a_small = desc_kmajor_sw128(cv + Cfg::TILE_BYTES + kk * 32);
          const uint64_t b_big = desc_kmajor_sw128(cv + 2 * Cfg::TILE_BYTES + kk * 32);
          const uint64_t b_small = desc_kmajor_sw128(cv + 3 * Cfg::TILE_BYTES + kk * 32);
          mma_tf32(d, a_small, b_big, Cfg::IDESC, (kt > kc0 || kk > 0) ? 1u : 0u);
          mma_tf32(d, a_big, b_small, Cfg::IDESC, 1u);
          mma_tf32(d, a_big, b_big, Cfg::IDESC, 1u);
        }
        mma_commit(bar.conv_empty(cs));  // frees the converted stage when these MMAs finish
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
template <class Cfg>
__device__ __forceinline__ void tc_epilogue(const TcParams &p, uint32_t tmem_base,
                                            const TcBars<Cfg> &bar, int q, int lane) {
  uint32_t chunk_iter = 0;
  const bool read_c = p.beta != 0.0f;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    float acc[Cfg::BN];  // this thread's row of the tile, FP32 round-to-nearest sums
#pragma unroll
    for (int j = 0; j < Cfg::BN; ++j) acc[j] = 0.0f;
    for (int kc0 = 0; kc0 < p.k_tiles; kc0 += Cfg::CHUNK_KTILES, ++chunk_iter) {
      const uint32_t b = chunk_iter & 1, use = chunk_iter >> 1;
      if (!wait_parity_bounded(bar.acc_full(b), use & 1, p.wait_budget_ns, p.status)) return;
      tc_fence_after_sync();
#pragma unroll
      for (int cc = 0; cc < Cfg::BN / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + b * 128 + cc * 32, v);
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
    const int row = tm * Cfg::BM + 32 * q + lane;
    const int n0 = tn * Cfg::BN;
    if (row < p.M) {
      float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int j = 0; j < Cfg::BN; j += 4) {
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
              crow[n + e] = read_c ? fmaf(p.alpha, acc[j + e], p.beta * crow[n + e])
                                   : p.alpha * acc[j + e];
        }
      }
    }
  }
}

// ------------------------------------------------------------------ kernel
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc3_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const TcBars<Cfg> bar{sbase + Cfg::BAR_OFFSET};
  const uint32_t tmem_slot = sbase + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::RAW_STAGES; ++s) {
      mbar_init(bar.raw_full(s), 1);
      mbar_init(bar.raw_empty(s), Cfg::CONVERTER_WARPS);
    }
    for (int s = 0; s < Cfg::CONV_STAGES; ++s) {
      mbar_init(bar.conv_full(s), Cfg::CONVERTER_WARPS);
      mbar_init(bar.conv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.acc_full(b), 1);
      mbar_init(bar.acc_empty(b), Cfg::EPILOGUE_WARPS);
    }
    mbar_init(bar.drain(), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base =
      *reinterpret_cast<volatile uint32_t *>(smem + Cfg::BAR_OFFSET + Cfg::NUM_BARS * 8);

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_WG0));
    if (warp == 0) {
      if (lane == 0) tc_produce<Cfg>(p, &tmA, &tmB, sbase, bar);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) tc_issue<Cfg>(p, sbase, tmem_base, bar);
      __syncwarp();
    }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_EPI));
    tc_epilogue<Cfg>(p, tmem_base, bar, warp & 3, lane);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REGS_CONV));
    tc_convert<Cfg>(p, smem, bar, threadIdx.x - 256, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace sg
