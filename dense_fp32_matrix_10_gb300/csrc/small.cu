// small.cu -- small and skinny products (SGEMM_ALGO_SMALL).
//
// The persistent kernels reach the FP32 peak on large products, but a
// product of a few tens of MFLOP is a chain of latencies there: the launch,
// the first TMA round trip, a k-slice or two per CTA and the stream-K pass
// that adds the split tiles' partial sums.  This kernel is one launch with
// no workspace: one CTA per 32 x 32 tile of C, K staged through shared
// memory in passes of 256 and split across the CTA's eight warps (32 k each
// per pass); the warps' partial tiles are then added in shared memory in warp
// order, so the result is deterministic.  Operands are read element by
// element along their stored layout (coalesced for either op, any alignment
// and leading dimension); each lane holds a 4 x 8 register tile of its warp's
// partial 32 x 32 tile (the register blocking of
// "CUDA矩阵乘法性能优化实战：从朴素内核到寄存器分块与Nsight剖析", section 5.2).
#include <mutex>

#include "internal.h"

namespace sg {
namespace {

constexpr int kTile = 32;        // C tile edge
constexpr int kWarps = 8;        // K split across the CTA's warps
constexpr int kThreads = 32 * kWarps;
constexpr int kPassK = 256;      // k staged per pass: kWarps x 32
constexpr int kStageFloats = kPassK * kTile;   // one operand's staged slice
constexpr int kSmemBytes = 2 * kStageFloats * 4;   // 64 KiB (the partial tiles reuse it)

// Float index of element (k, j) of a staged [kPassK][32] slice: 16-byte
// chunk (j / 4) XOR (k mod 8), so that column-wise staging writes and the
// compute loop's float4 reads spread over the banks.
__device__ __forceinline__ int swz(int k, int j) {
  return k * kTile + ((((j >> 2) ^ (k & 7)) << 2) | (j & 3));
}

__global__ void __launch_bounds__(kThreads, 2)
    small_gemm_kernel(const PlainParams p) {
  extern __shared__ __align__(16) float smem[];
  float *As = smem;                 // As[k][m]: op(A) rows m0 .. m0+31
  float *Bs = smem + kStageFloats;  // Bs[k][n]: op(B) columns n0 .. n0+31
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int tr = lane >> 2, tc = lane & 3;   // rows 4tr..4tr+3, columns 8tc..8tc+7
  float2 acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[r][q] = make_float2(0.0f, 0.0f);

  for (int k0 = 0; k0 < p.K; k0 += kPassK) {
    // ---- stage op(A)[m0.., k0..] and op(B)[k0.., n0..]; zeros outside.
    // Pass `it` of a thread covers, in the stored layout's contiguous
    // direction, 256 consecutive k (k-contiguous operand: one row/column of
    // the tile per pass) or eight k of 32 consecutive m/n; the passes' loads
    // are independent, sixteen of them in flight at once.
#pragma unroll 16
    for (int it = 0; it < kStageFloats / kThreads; ++it) {
      const int k = p.transA == 0 ? t : it * (kThreads / kTile) + (t >> 5);
      const int j = p.transA == 0 ? it : (t & 31);
      const int gm = m0 + j, gk = k0 + k;
      float v = 0.0f;
      if (gm < p.M && gk < p.K)
        v = p.transA == 0 ? p.A[static_cast<int64_t>(gm) * p.lda + gk]
                          : p.A[static_cast<int64_t>(gk) * p.lda + gm];
      As[swz(k, j)] = v;
    }
#pragma unroll 16
    for (int it = 0; it < kStageFloats / kThreads; ++it) {
      const int k = p.transB == 1 ? t : it * (kThreads / kTile) + (t >> 5);
      const int j = p.transB == 1 ? it : (t & 31);
      const int gn = n0 + j, gk = k0 + k;
      float v = 0.0f;
      if (gn < p.N && gk < p.K)
        v = p.transB == 0 ? p.B[static_cast<int64_t>(gk) * p.ldb + gn]
                          : p.B[static_cast<int64_t>(gn) * p.ldb + gk];
      Bs[swz(k, j)] = v;
    }
    __syncthreads();
    // ---- this warp's 32 k of the pass, in ascending order
    const int kw = warp * 32;
    const int kend = min(32, p.K - k0 - kw);   // <= 0: nothing of this pass
#pragma unroll 4
    for (int kk = 0; kk < kend; ++kk) {
      const int k = kw + kk;
      const float4 a = *reinterpret_cast<const float4 *>(&As[swz(k, 4 * tr)]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[swz(k, 8 * tc)]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[swz(k, 8 * tc + 4)]);
      const float ar[4] = {a.x, a.y, a.z, a.w};
      const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                            make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          acc[r][q] = __ffma2_rn(make_float2(ar[r], ar[r]), bp[q], acc[r][q]);
    }
    __syncthreads();   // the slices are overwritten by the next pass
  }

  // ---- partial tiles of the eight warps, added in warp order
  float *part = smem;   // [kWarps][32][32]
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<float2 *>(&part[(warp * kTile + 4 * tr + r) * kTile + 8 * tc + 2 * q]) =
          acc[r][q];
  __syncthreads();
  for (int o = t; o < kTile * kTile; o += kThreads) {
    const int row = m0 + o / kTile, col = n0 + o % kTile;
    float s = part[o];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) s += part[w * kTile * kTile + o];
    if (row < p.M && col < p.N) {
      float *c = p.C + static_cast<int64_t>(row) * p.ldc + col;
      *c = p.beta == 0.0f ? p.alpha * s : fmaf(p.alpha, s, p.beta * *c);
    }
  }
}

}  // namespace

cudaError_t launch_small(const PlainParams &p, cudaStream_t s) {
  static_assert(kWarps * kTile * kTile <= 2 * kStageFloats, "partial tiles exceed the staging");
  const int64_t gy = (static_cast<int64_t>(p.M) + kTile - 1) / kTile;
  const int64_t gx = (static_cast<int64_t>(p.N) + kTile - 1) / kTile;
  if (gy > 65535 || gx > 2147483647) return cudaErrorInvalidValue;
  // the 64 KiB of dynamic shared memory, once per device
  constexpr int kMaxDevices = 64;
  static std::once_flag once[kMaxDevices];
  static cudaError_t attr[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [dev]() {
    attr[dev] = cudaFuncSetAttribute(small_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
  });
  if (attr[dev] != cudaSuccess) return attr[dev];
  small_gemm_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kThreads, kSmemBytes,
                      s>>>(p);
  return cudaGetLastError();
}

}  // namespace sg
