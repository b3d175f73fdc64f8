// internal.h -- declarations shared by the library's translation units
// (host side).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "simt_gemm.cuh"
#include "tc_3xtf32.cuh"

namespace sg {

// Tile configurations of the CUDA-core kernels (8 x 8 outputs per thread,
// 32 x 64 per warp).
enum SimtTile : int {
  kTile128x128 = 0,  // 4 x 2 math warps, 8 x 8 per thread
  kTile128x64 = 1,   // 4 x 1 math warps, 8 x 8 per thread (two CTAs per SM)
  kTile128x256 = 2,  // 4 x 2 math warps, 8 x 16 per thread (n-contiguous op(B) only)
  kNumSimtTiles = 3
};

// Launches `kernel`; with `pdl` it may be scheduled before the previous
// kernel on the stream has finished (the kernel must call griddep_wait()
// before touching memory that kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// As launch_maybe_pdl, in clusters of `cluster` CTAs along x when cluster > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t s, bool pdl, int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

struct SimtKernelInfo {
  int bm, bn, threads, smem_bytes, ctas_per_sm;
  // clusters of 2, 4 and 8 CTAs resident at once on the device (0: that
  // cluster size cannot be launched)
  int max_clusters[3];
};

// Launches one instantiation; grid = number of CTAs (persistent, or S per
// tile with cluster split-K).
// pdl: launch with programmatic stream serialization (it directly follows
// another kernel of the same call on the stream).  cluster: CTAs per cluster
// along x (1: no cluster).
using SimtLaunchFn = cudaError_t (*)(const SimtParams &, const CUtensorMap *, const CUtensorMap *,
                                     const CUtensorMap *, int grid, cudaStream_t, bool pdl,
                                     int cluster);
// Sets the kernel's shared-memory attribute on the current device (once) and
// reports its shape and occupancy.
using SimtInfoFn = cudaError_t (*)(SimtKernelInfo *);

struct SimtEntry {
  SimtLaunchFn launch;
  SimtInfoFn info;
};

// [producer][transA][transB][tile]; csk: the cluster split-K form (128 x 128
// and 128 x 64 tiles)
SimtEntry simt_entry(int producer, int transA, int transB, int tile, int csk = 0);

// 3xTF32 tensor-core kernel (tc_3xtf32.cu), 128 x 128 tiles, one CTA per SM.
struct TcKernelInfo {
  int bm, bn, ctas_per_sm;
  int max_ctas;   // CTAs of this kernel resident at once on the device
};
// Maps: op(A), op(B), and -- for the pre-split form only -- A's and B's small
// parts (K-major); the other forms ignore the last two.
using TcLaunchFn = cudaError_t (*)(const TcParams &, const CUtensorMap *, const CUtensorMap *,
                                   const CUtensorMap *, const CUtensorMap *, int, cudaStream_t,
                                   bool pdl);
using TcInfoFn = cudaError_t (*)(TcKernelInfo *);
struct TcEntry {
  TcLaunchFn launch;
  TcInfoFn info;
};
TcEntry tc3_entry(int transA, int transB);
// The form that reads pre-split operands: A and B k-contiguous big parts plus
// their small parts, all through TMA (no conversion in the kernel).
// bn = 128 or 256: the output tile width.
TcEntry tc3_presplit_entry(int bn);
// The same product on CTA pairs (256 x bn tiles, bn = 128 or 256, launched
// in clusters of two; grid = 2 x the pair count, p.tiles_m counting 256-row
// tile rows).  fold_a / fold_b: that operand is k-contiguous and its small
// parts are computed in the kernel (its big-part map is the operand itself;
// its small-part map is not read).
TcEntry tc3_pair_entry(int bn, bool fold_a = false, bool fold_b = false);

// Second pass of a stream-K launch (sk_fixup.cu).
// load_sk_fixup / load_scale_c: make the CUDA runtime load these kernels now
// (under lazy module loading it would do so at their first launch).
cudaError_t load_sk_fixup();
cudaError_t load_scale_c();
cudaError_t launch_sk_fixup(const SimtParams &p, int bm, int bn, int grid_main, int sk_tiles,
                            int sm_count, cudaStream_t s);

// Context kernels and helpers (context.cu).
struct PlainParams {
  const float *A;
  const float *B;
  float *C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  int transA, transB;
  float alpha, beta;
  int *status = nullptr;   // device status word (debug-bounds builds report here)
};
cudaError_t launch_naive(const PlainParams &p, cudaStream_t s);
cudaError_t launch_smem_tiled(const PlainParams &p, cudaStream_t s);
// Register-tiled comparison kernel, R x R outputs per thread (R = 2 or 4).
cudaError_t launch_reg_tiled(const PlainParams &p, int R, cudaStream_t s);
// SGEMM_ALGO_SMALL (small.cu); cudaErrorInvalidValue if M needs more than
// 65535 row tiles.
cudaError_t launch_small(const PlainParams &p, cudaStream_t s);
cudaError_t launch_scale_c(float *C, int64_t ldc, int M, int N, float beta, cudaStream_t s);
// out (cols x rows, ld_out) = in (rows x cols, ld_in) transposed (transpose.cu);
// `status` is the device status word the bounded waits report to.  Unless
// exact_edges, up to three floats past the end of each output row (inside
// ld_out rounded up to 4) may be written too (library scratch).
cudaError_t launch_transpose(const float *in, int64_t ld_in, float *out, int64_t ld_out, int rows,
                             int cols, int sm_count, int *status, cudaStream_t s, bool exact_edges = false);
// The split pass of the 3xTF32 product (transpose.cu): the TF32 small parts of
// a rows x cols operand (k along each row when !transpose, down the columns
// when transpose), written K-major to `small` (ld_out); with `transpose` the
// operand is also written transposed to `big` (its TF32 big parts).  *done is false when the pass
// could not run (then nothing was queued).
cudaError_t launch_tf32_split(const float *in, int64_t ld_in, int rows, int cols, bool transpose,
                              float *big, float *small, int64_t ld_out, int sm_count, int *status,
                              cudaStream_t s, bool *done);
cudaError_t launch_scale_c_batched(float *C, int64_t ldc, int64_t strideC, int M, int N,
                                   int64_t batch, float beta, cudaStream_t s);
cudaError_t launch_wait_selftest(uint64_t budget_ns, int *status, cudaStream_t s);

}  // namespace sg
