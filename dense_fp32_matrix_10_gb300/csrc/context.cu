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
