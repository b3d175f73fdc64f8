// simt_instances.cuh -- defines launch/info wrappers for one family of
// instantiations of the CUDA-core kernel.  Included by the simt_*.cu units,
// each of which fixes PRODUCER and TRANS_A to keep translation units small
// (they compile in parallel).
#pragma once

#include "internal.h"

namespace sg {

template <class Cfg>
cudaError_t simt_launch(const SimtParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                        const CUtensorMap *tmC, int grid, cudaStream_t stream, bool pdl, int cluster) {
  return launch_cluster_maybe_pdl(simt_gemm_kernel<Cfg>, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES,
                                  stream, pdl, cluster, *tmA, *tmB, *tmC, p);
}

template <class Cfg>
cudaError_t simt_info(SimtKernelInfo *info) {
  cudaError_t e = cudaFuncSetAttribute(simt_gemm_kernel<Cfg>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the CTA's launch registers can cover the new
  // split; refuse to launch a build whose launch register count is too small.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, simt_gemm_kernel<Cfg>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * Cfg::THREADS <
      Cfg::PRODUCER_THREADS * Cfg::PRODUCER_REGS + Cfg::MATH_THREADS * Cfg::MATH_REGS)
    return cudaErrorInvalidConfiguration;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, simt_gemm_kernel<Cfg>, Cfg::THREADS,
                                                    Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  info->bm = Cfg::BM;
  info->bn = Cfg::BN;
  info->threads = Cfg::THREADS;
  info->smem_bytes = Cfg::SMEM_BYTES;
  info->ctas_per_sm = occ;
  // clusters of 2, 4, 8 CTAs (cluster split-K) that fit at once: a cluster
  // needs its CTAs on SMs of one GPC
  for (int i = 0; i < 3; ++i) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 << i);
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 << i;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, simt_gemm_kernel<Cfg>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
    info->max_clusters[i] = clusters;
  }
  return cudaSuccess;
}

template <int PRODUCER, bool A_KMAJOR, bool B_KMAJOR, int TILE, bool CSK>
struct SimtPick;
// With the TMA producer a k-contiguous A is transposed in shared memory
// (SG_SIMT_TRANSPOSE_A).
template <int PRODUCER, bool A_KMAJOR>
constexpr bool kTransA = (PRODUCER == kTma) && A_KMAJOR && SG_SIMT_TRANSPOSE_A;

template <int PRODUCER, bool A_KMAJOR, bool B_KMAJOR, bool CSK>
struct SimtPick<PRODUCER, A_KMAJOR, B_KMAJOR, kTile128x128, CSK> {
  using Cfg = SimtConfig<4, 2, A_KMAJOR, B_KMAJOR, 4, PRODUCER, 8, kTransA<PRODUCER, A_KMAJOR>, CSK>;
};
// 128 x 64 tiles run two CTAs per SM.  With the raw A ring of the in-smem
// transpose (32 KiB) four stages would need ~129 KiB per CTA, and only one
// CTA -- four math warps -- would fit on an SM; three stages (~105 KiB) let
// two fit.
#ifndef SG_SIMT_STAGES_64_TRANS
#define SG_SIMT_STAGES_64_TRANS 3
#endif
template <int PRODUCER, bool A_KMAJOR, bool B_KMAJOR, bool CSK>
struct SimtPick<PRODUCER, A_KMAJOR, B_KMAJOR, kTile128x64, CSK> {
  static constexpr bool kT = kTransA<PRODUCER, A_KMAJOR>;
  using Cfg = SimtConfig<4, 1, A_KMAJOR, B_KMAJOR, kT ? SG_SIMT_STAGES_64_TRANS : 4, PRODUCER, 8, kT, CSK>;
  static_assert(2 * (Cfg::SMEM_BYTES + 1024) <= 233472, "two 128 x 64 CTAs must fit on an SM");
};
template <int PRODUCER, bool A_KMAJOR, bool CSK>
struct SimtPick<PRODUCER, A_KMAJOR, false, kTile128x256, CSK> {
  using Cfg = SimtConfig<4, 2, A_KMAJOR, false, 4, PRODUCER, 16, kTransA<PRODUCER, A_KMAJOR>, CSK>;
};

template <int PRODUCER, bool A_KMAJOR, bool B_KMAJOR, int TILE, bool CSK = false>
SimtEntry simt_make_entry() {
  using Cfg = typename SimtPick<PRODUCER, A_KMAJOR, B_KMAJOR, TILE, CSK>::Cfg;
  return SimtEntry{&simt_launch<Cfg>, &simt_info<Cfg>};
}

// A stored M x K (transA = N) is the k-contiguous ("K-major") layout; B stored
// N x K (transB = T) likewise.
// The 128 x 256 tile exists only for n-contiguous op(B) (transB = N) and the
// TMA producer (the only combination the dispatcher picks it for); any other
// request for it gets the 128 x 128 tile.  The cluster split-K form (csk)
// exists for the 128 x 128 and 128 x 64 tiles.
#define SG_DEFINE_SIMT_FAMILY(PROD, TA)                                                  \
  SimtEntry simt_entry_##PROD##_##TA(int transB, int tile, int csk) {                    \
    constexpr bool AK = (TA == 0);                                                       \
    if (csk) {                                                                           \
      if (transB == 0)                                                                   \
        return tile == kTile128x64 ? simt_make_entry<PROD, AK, false, kTile128x64, true>() \
                                   : simt_make_entry<PROD, AK, false, kTile128x128, true>(); \
      return tile == kTile128x64 ? simt_make_entry<PROD, AK, true, kTile128x64, true>()  \
                                 : simt_make_entry<PROD, AK, true, kTile128x128, true>(); \
    }                                                                                    \
    if (transB == 0) {                                                                   \
      if constexpr (PROD == kTma)                                                        \
        if (tile == kTile128x256) return simt_make_entry<PROD, AK, false, kTile128x256>(); \
      return tile == kTile128x128 ? simt_make_entry<PROD, AK, false, kTile128x128>()     \
                                  : simt_make_entry<PROD, AK, false, kTile128x64>();      \
    }                                                                                    \
    return tile == kTile128x64 ? simt_make_entry<PROD, AK, true, kTile128x64>()          \
                               : simt_make_entry<PROD, AK, true, kTile128x128>();        \
  }

}  // namespace sg
