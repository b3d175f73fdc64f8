// context.cu -- the comparison kernels of the pages, re-written for the
// general op/ld/alpha/beta form, plus two small helpers of the dispatcher.
//
//  * naive_kernel: one thread per output, every operand read straight from
//    global memory -- the first kernel of
//    "CUDA矩阵乘法性能优化实战：从朴素内核到寄存器分块与Nsight剖析" (section 2.1),
//    16 x 16 thread blocks as there.
//  * smem_tiled_kernel: 16 x 16 output tile per block, one output per thread,
//    op(A)/op(B) 16 x 16 tiles staged in shared memory with one column of
//    padding and zero-filled edges, two barriers per k step -- the second
//    kernel of the same article (sections 3.2, 3.3).
//  * reg_tiled_kernel<R>: 16 x 16 threads, each holding an R x R block of
//    outputs in registers (R = 2 or 4, a (16R) x (16R) tile per block), so
//    that every value read from shared memory feeds R multiply-adds; the
//    operands move in R-wide vector loads (float2 / float4) wherever alignment
//    and the matrix edge allow -- the third rung of the same article
//    (sections 5.2 and 5.3: register tiling, float4 loads, __restrict__).
//  * scale_c_kernel: C = beta * C (beta == 0 writes zeros without reading C),
//    the whole result when K == 0 or alpha == 0.
//  * wait_selftest_kernel: waits, with the library's bounded wait, on an
//    mbarrier that never completes, so the give-up path can be observed.
#include "internal.h"

namespace sg {

__device__ __forceinline__ float load_opA(const PlainParams &p, int i, int k) {
  return p.transA ? p.A[static_cast<int64_t>(k) * p.lda + i] : p.A[static_cast<int64_t>(i) * p.lda + k];
}
__device__ __forceinline__ float load_opB(const PlainParams &p, int k, int j) {
  return p.transB ? p.B[static_cast<int64_t>(j) * p.ldb + k] : p.B[static_cast<int64_t>(k) * p.ldb + j];
}

__device__ __forceinline__ void store_out(const PlainParams &p, int i, int j, float acc) {
  float *c = p.C + static_cast<int64_t>(i) * p.ldc + j;
  *c = (p.beta != 0.0f) ? fmaf(p.alpha, acc, p.beta * *c) : p.alpha * acc;
}

__global__ void naive_kernel(const PlainParams p) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y * blockDim.y + threadIdx.y;
  if (i >= p.M || j >= p.N) return;
  float acc = 0.0f;
  for (int k = 0; k < p.K; ++k) acc = fmaf(load_opA(p, i, k), load_opB(p, k, j), acc);
  store_out(p, i, j, acc);
}

constexpr int kT = 16;

__global__ void smem_tiled_kernel(const PlainParams p) {
  __shared__ float As[kT][kT + 1];
  __shared__ float Bs[kT][kT + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.y * kT + ty;
  const int j = blockIdx.x * kT + tx;
  float acc = 0.0f;
  for (int k0 = 0; k0 < p.K; k0 += kT) {
    As[ty][tx] = (i < p.M && k0 + tx < p.K) ? load_opA(p, i, k0 + tx) : 0.0f;
    Bs[ty][tx] = (k0 + ty < p.K && j < p.N) ? load_opB(p, k0 + ty, j) : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kT; ++k) acc = fmaf(As[ty][k], Bs[k][tx], acc);
    __syncthreads();
  }
  if (i < p.M && j < p.N) store_out(p, i, j, acc);
}

// ---- register-tiled rung
// Shared tiles are k-major (As[k][m], Bs[k][n]) so that a thread's R values of
// op(A) and of op(B) at one k are adjacent: one vector shared load each, then
// R * R multiply-adds.  k is walked in slices of 16; every thread stages R
// consecutive elements of each operand per slice, along the stored layout's
// contiguous direction (whole 64-byte row pieces per four threads when k is
// contiguous), transposing into the k-major tile where needed.
template <int R> struct RegVec;
template <> struct RegVec<2> {
  using type = float2;
  static __device__ __forceinline__ float2 make(const float (&v)[2]) { return make_float2(v[0], v[1]); }
};
template <> struct RegVec<4> {
  using type = float4;
  static __device__ __forceinline__ float4 make(const float (&v)[4]) {
    return make_float4(v[0], v[1], v[2], v[3]);
  }
};

// R consecutive floats from src: one vector load when `vec` (the run is
// aligned) and all R lie inside the matrix (avail >= R), else element by
// element, zeros past `avail`.
template <int R>
__device__ __forceinline__ void load_run(const float *__restrict__ src, bool vec, int avail, float (&v)[R]) {
  using V = typename RegVec<R>::type;
  if (vec && avail >= R) {
    const V x = __ldg(reinterpret_cast<const V *>(src));
    const float *f = reinterpret_cast<const float *>(&x);
#pragma unroll
    for (int q = 0; q < R; ++q) v[q] = f[q];
  } else {
#pragma unroll
    for (int q = 0; q < R; ++q) v[q] = q < avail ? src[q] : 0.0f;
  }
}

constexpr int kRegBK = 16;

// Stages the kRegBK x (16R) slice starting at (k0, x0) of op(X) into Xs[k][x]
// (X = A with x = m, or X = B with x = n).  kcontig: X stored with k along its
// rows (op(A) = N, op(B) = T), else x along its rows.
template <int R>
__device__ __forceinline__ void stage_slice(const float *__restrict__ X, int64_t ld, bool kcontig, bool vec,
                                            int xdim, int K, int x0, int k0, int t,
                                            float (&Xs)[kRegBK][16 * R]) {
  constexpr int W = 16 * R;
  float v[R];
  if (kcontig) {   // W rows of 16 k each: 16 / R runs per row
    const int x = t / (kRegBK / R), kr = (t % (kRegBK / R)) * R;
    const int gx = x0 + x, gk = k0 + kr;
    const int avail = gx < xdim ? min(R, K - gk) : 0;
    load_run<R>(X + static_cast<int64_t>(gx < xdim ? gx : 0) * ld + (gk < K ? gk : 0), vec, avail, v);
#pragma unroll
    for (int q = 0; q < R; ++q) Xs[kr + q][x] = v[q];
  } else {         // 16 k-rows of W: W / R runs per k-row
    const int kr = t / (W / R), x = (t % (W / R)) * R;
    const int gk = k0 + kr, gx = x0 + x;
    const int avail = gk < K ? min(R, xdim - gx) : 0;
    load_run<R>(X + static_cast<int64_t>(gk < K ? gk : 0) * ld + (gx < xdim ? gx : 0), vec, avail, v);
    using V = typename RegVec<R>::type;
    *reinterpret_cast<V *>(&Xs[kr][x]) = RegVec<R>::make(v);
  }
}

// vec: bit 0 op(A) runs, bit 1 op(B) runs, bit 2 C rows may use R-wide vectors
// (base aligned to 4R bytes, leading dimension a multiple of R).
template <int R>
__global__ void __launch_bounds__(256) reg_tiled_kernel(const PlainParams p, int vec) {
  constexpr int W = 16 * R;
  __shared__ __align__(16) float As[kRegBK][W];
  __shared__ __align__(16) float Bs[kRegBK][W];
  using V = typename RegVec<R>::type;
  const int tx = threadIdx.x, ty = threadIdx.y, t = ty * 16 + tx;
  const int m0 = blockIdx.y * W, n0 = blockIdx.x * W;
  float acc[R][R];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < R; ++c) acc[r][c] = 0.0f;
  for (int k0 = 0; k0 < p.K; k0 += kRegBK) {
    stage_slice<R>(p.A, p.lda, p.transA == 0, vec & 1, p.M, p.K, m0, k0, t, As);
    stage_slice<R>(p.B, p.ldb, p.transB == 1, vec & 2, p.N, p.K, n0, k0, t, Bs);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRegBK; ++k) {
      const V av = *reinterpret_cast<const V *>(&As[k][ty * R]);
      const V bv = *reinterpret_cast<const V *>(&Bs[k][tx * R]);
      const float *a = reinterpret_cast<const float *>(&av);
      const float *b = reinterpret_cast<const float *>(&bv);
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < R; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
  const int j0 = n0 + tx * R;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = m0 + ty * R + r;
    if (i >= p.M) break;
    if ((vec & 4) && j0 + R <= p.N) {
      V *c = reinterpret_cast<V *>(p.C + static_cast<int64_t>(i) * p.ldc + j0);
      V o;
      float *f = reinterpret_cast<float *>(&o);
      if (p.beta != 0.0f) {
        const V old = *c;
        const float *g = reinterpret_cast<const float *>(&old);
#pragma unroll
        for (int q = 0; q < R; ++q) f[q] = fmaf(p.alpha, acc[r][q], p.beta * g[q]);
      } else {
#pragma unroll
        for (int q = 0; q < R; ++q) f[q] = p.alpha * acc[r][q];
      }
      *c = o;
    } else {
#pragma unroll
      for (int q = 0; q < R; ++q)
        if (j0 + q < p.N) store_out(p, i, j0 + q, acc[r][q]);
    }
  }
}

// C_b = beta * C_b for b < batch (C_b = C + b * strideC).
__global__ void scale_c_kernel(float *C, int64_t ldc, int64_t strideC, int M, int N, int64_t batch,
                               float beta) {
  const int64_t per = static_cast<int64_t>(M) * N, total = per * batch;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = e / per, r = e - b * per;
    const int64_t i = r / N, j = r - i * N;
    float *c = C + b * strideC + i * ldc + j;
    *c = (beta != 0.0f) ? beta * *c : 0.0f;
  }
}

__global__ void wait_selftest_kernel(uint64_t budget_ns, int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  // Nothing arrives: the bounded wait must give up and record the timeout.
  wait_parity_bounded(b, 0, budget_ns, status);
}

cudaError_t launch_naive(const PlainParams &p, cudaStream_t s) {
  dim3 block(16, 16);
  dim3 grid((p.N + 15) / 16, (p.M + 15) / 16);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  naive_kernel<<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_smem_tiled(const PlainParams &p, cudaStream_t s) {
  dim3 block(kT, kT);
  dim3 grid((p.N + kT - 1) / kT, (p.M + kT - 1) / kT);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  smem_tiled_kernel<<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

// R-wide vector accesses to a matrix need its base aligned to 4R bytes and
// its leading dimension a multiple of R.
static bool vec_ok(const void *base, int64_t ld, int R) {
  return reinterpret_cast<uintptr_t>(base) % (4 * R) == 0 && ld % R == 0;
}

cudaError_t launch_reg_tiled(const PlainParams &p, int R, cudaStream_t s) {
  const int W = 16 * R;
  dim3 block(16, 16);
  dim3 grid((p.N + W - 1) / W, (p.M + W - 1) / W);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const int vec = (vec_ok(p.A, p.lda, R) ? 1 : 0) | (vec_ok(p.B, p.ldb, R) ? 2 : 0) |
                  (vec_ok(p.C, p.ldc, R) ? 4 : 0);
  if (R == 2)
    reg_tiled_kernel<2><<<grid, block, 0, s>>>(p, vec);
  else
    reg_tiled_kernel<4><<<grid, block, 0, s>>>(p, vec);
  return cudaGetLastError();
}

cudaError_t load_scale_c() {
  cudaFuncAttributes attr;
  return cudaFuncGetAttributes(&attr, scale_c_kernel);
}

cudaError_t launch_scale_c(float *C, int64_t ldc, int M, int N, float beta, cudaStream_t s) {
  return launch_scale_c_batched(C, ldc, 0, M, N, 1, beta, s);
}

cudaError_t launch_scale_c_batched(float *C, int64_t ldc, int64_t strideC, int M, int N,
                                   int64_t batch, float beta, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(M) * N * batch;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond 16 waves of 152 SMs
  scale_c_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(C, ldc, strideC, M, N, batch, beta);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t budget_ns, int *status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 1, 0, s>>>(budget_ns, status);
  return cudaGetLastError();
}

}  // namespace sg
