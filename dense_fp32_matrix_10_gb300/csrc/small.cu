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
#include "ptx.cuh"

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

// Stages the 32 rows r0 .. r0+31 of an operand panel (op(A)'s rows or
// op(B)'s columns), k in [k0, k0 + 256), into S (swizzled [k][32]); zeros
// outside [0, R) x [0, K).  KCONTIG: the stored rows run along k
// (X[r * ld + k]), else along r (X[k * ld + r]).  A panel wholly inside the
// matrix with 16-byte aligned rows is read as float4, every load issued
// before any store; the rest element by element with predicated loads.
// Either way a warp reads along the stored rows.
template <bool KCONTIG>
__device__ __forceinline__ void stage_panel(const float *__restrict__ X, int64_t ld, int R, int K,
                                            int r0, int k0, float *S, int t) {
  constexpr int kVecIters = kStageFloats / (4 * kThreads);   // 8 float4 per thread
  const bool vec = (ld % 4 == 0) && ((reinterpret_cast<uintptr_t>(X) & 15) == 0) &&
                   r0 + kTile <= R && k0 + kPassK <= K;
  if (vec) {
    float4 v[kVecIters];
    if (KCONTIG) {
      // a warp covers 8 rows x 16 k: 64-byte row segments, stores spread
      // over 16 banks
      const int lane = t & 31, w = t >> 5;
      const int j = (w & 3) * 8 + (lane & 7);
      const int qb = (w >> 2) * 4 + (lane >> 3);
      const float *src = X + static_cast<int64_t>(r0 + j) * ld + k0 + 4 * qb;
#pragma unroll
      for (int it = 0; it < kVecIters; ++it) v[it] = *reinterpret_cast<const float4 *>(src + 32 * it);
#pragma unroll
      for (int it = 0; it < kVecIters; ++it) {
        const int q = it * 8 + qb;
        S[swz(4 * q, j)] = v[it].x;
        S[swz(4 * q + 1, j)] = v[it].y;
        S[swz(4 * q + 2, j)] = v[it].z;
        S[swz(4 * q + 3, j)] = v[it].w;
      }
    } else {
      // a warp covers 4 k x 32 rows: 128-byte row segments, one 16-byte
      // chunk of S per lane
      const int q = t & 7, kb = t >> 3;
      const float *src = X + static_cast<int64_t>(k0 + kb) * ld + r0 + 4 * q;
#pragma unroll
      for (int it = 0; it < kVecIters; ++it)
        v[it] = *reinterpret_cast<const float4 *>(src + static_cast<int64_t>(32 * it) * ld);
#pragma unroll
      for (int it = 0; it < kVecIters; ++it)
        *reinterpret_cast<float4 *>(&S[swz(it * 32 + kb, 4 * q)]) = v[it];
    }
    return;
  }
  // element by element: consecutive lanes take consecutive elements of a
  // stored row (256 k of one row, or 32 rows of eight k)
#pragma unroll 16
  for (int it = 0; it < kStageFloats / kThreads; ++it) {
    const int k = KCONTIG ? t : it * (kThreads / kTile) + (t >> 5);
    const int j = KCONTIG ? it : (t & 31);
    const int r = r0 + j, gk = k0 + k;
    float v = 0.0f;
    if (r < R && gk < K)
      v = KCONTIG ? X[static_cast<int64_t>(r) * ld + gk] : X[static_cast<int64_t>(gk) * ld + r];
    S[swz(k, j)] = v;
  }
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
  // launched as a programmatic dependent of the stream's previous kernel:
  // A, B and C are touched only once that kernel has completed
  griddep_wait();

  for (int k0 = 0; k0 < p.K; k0 += kPassK) {
    // ---- stage op(A)[m0.., k0..] and op(B)[k0.., n0..]; zeros outside
    if (p.transA == 0)
      stage_panel<true>(p.A, p.lda, p.M, p.K, m0, k0, As, t);
    else
      stage_panel<false>(p.A, p.lda, p.M, p.K, m0, k0, As, t);
    if (p.transB == 1)
      stage_panel<true>(p.B, p.ldb, p.N, p.K, n0, k0, Bs, t);
    else
      stage_panel<false>(p.B, p.ldb, p.N, p.K, n0, k0, Bs, t);
    __syncthreads();
    // ---- this warp's 32 k of the pass, in ascending order
    const int kw = warp * 32;
    const int kend = min(32, p.K - k0 - kw);   // <= 0: nothing of this pass
#pragma unroll 4
    for (int kk = 0; kk < kend; ++kk) {
      const int k = kw + kk;
      if (!SG_CHECK(k < kPassK && swz(k, 8 * tc + 4) + 4 <= kStageFloats, p.status)) break;
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

  // the next kernel on the stream may be scheduled (it waits for this one
  // to complete before touching memory)
  griddep_launch_dependents();

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
    if (!SG_CHECK(o + (kWarps - 1) * kTile * kTile < 2 * kStageFloats, p.status)) break;
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
  // programmatic stream serialization: back-to-back small products overlap
  // one kernel's launch with the previous one's tail
  return launch_maybe_pdl(small_gemm_kernel,
                          dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(kThreads),
                          kSmemBytes, s, true, p);
}

}  // namespace sg
