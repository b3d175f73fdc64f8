// Instantiations and host launch wrappers of the 3xTF32 tensor-core kernel
// (one per op(A) / op(B) layout).
#include "internal.h"
#include "tc_3xtf32.cuh"
#include "tc_3xtf32_pair.cuh"

namespace sg {

template <class Cfg>
static cudaError_t tc3_launch(const TcParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                              const CUtensorMap *tmAs, const CUtensorMap *tmBs, int grid,
                              cudaStream_t stream, bool pdl) {
  return launch_maybe_pdl(tc3_gemm_kernel<Cfg>, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES,
                          stream, pdl, *tmA, *tmB, *tmAs, *tmBs, p);
}

template <class Cfg>
static cudaError_t tc3_info(TcKernelInfo *info) {
  cudaError_t e = cudaFuncSetAttribute(tc3_gemm_kernel<Cfg>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the launch registers cover the split: refuse a
  // build whose launch register count is too small.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, tc3_gemm_kernel<Cfg>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * Cfg::THREADS < Cfg::REGS_SPLIT)
    return cudaErrorInvalidConfiguration;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, tc3_gemm_kernel<Cfg>, Cfg::THREADS,
                                                    Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  info->bm = Cfg::BM;
  info->bn = Cfg::BN;
  info->ctas_per_sm = occ;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  info->max_ctas = sms * occ;
  return cudaSuccess;
}

template <bool AK, bool BK, bool PRESPLIT = false, int BN = 128>
static TcEntry tc3_make() {
  using Cfg = TcConfig<AK, BK, PRESPLIT, BN>;
  return TcEntry{&tc3_launch<Cfg>, &tc3_info<Cfg>};
}

TcEntry tc3_presplit_entry(int bn) {
  return bn == 256 ? tc3_make<true, true, true, 256>() : tc3_make<true, true, true>();
}

// ---------------------------------------------------------------- CTA pairs
template <class Cfg>
static cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute *attr,
                                      bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

template <class Cfg>
static cudaError_t tc3_pair_launch(const TcParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB,
                                   const CUtensorMap *tmAs, const CUtensorMap *tmBs, int grid,
                                   cudaStream_t stream, bool pdl) {
  if (grid < 2 || grid % 2 != 0) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config<Cfg>(grid, stream, attr, pdl);
  return cudaLaunchKernelEx(&cfg, tc3_pair_kernel<Cfg>, *tmA, *tmB, *tmAs, *tmBs, p);
}

template <class Cfg>
static cudaError_t tc3_pair_info(TcKernelInfo *info) {
  cudaError_t e = cudaFuncSetAttribute(tc3_pair_kernel<Cfg>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the launch registers cover the split
  cudaFuncAttributes attr_k;
  e = cudaFuncGetAttributes(&attr_k, tc3_pair_kernel<Cfg>);
  if (e != cudaSuccess) return e;
  if (Cfg::EPILOGUE_GROUPS > 1 &&
      attr_k.numRegs * Cfg::THREADS < 128 * (Cfg::REGS_WG0 + 2 * Cfg::REGS_EPI))
    return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // a pair needs two free SMs of one GPC: ask how many pairs fit at once
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config<Cfg>(2 * sms, nullptr, attr, false);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, tc3_pair_kernel<Cfg>, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  info->bm = Cfg::BM;
  info->bn = Cfg::BN;
  info->ctas_per_sm = 1;
  info->max_ctas = 2 * clusters;
  return cudaSuccess;
}

template <int BN, bool FA, bool FB>
static TcEntry tc3_pair_make() {
  return TcEntry{&tc3_pair_launch<TcPairConfig<BN, FA, FB>>, &tc3_pair_info<TcPairConfig<BN, FA, FB>>};
}

TcEntry tc3_pair_entry(int bn, bool fold_a, bool fold_b) {
  if (bn == 256) {
    if (fold_a) return fold_b ? tc3_pair_make<256, true, true>() : tc3_pair_make<256, true, false>();
    return fold_b ? tc3_pair_make<256, false, true>() : tc3_pair_make<256, false, false>();
  }
  if (fold_a) return fold_b ? tc3_pair_make<128, true, true>() : tc3_pair_make<128, true, false>();
  return fold_b ? tc3_pair_make<128, false, true>() : tc3_pair_make<128, false, false>();
}

TcEntry tc3_entry(int transA, int transB) {
  // A stored M x K (transA = N) and B stored N x K (transB = T) are k-contiguous.
  if (transA == 0) return transB ? tc3_make<true, true>() : tc3_make<true, false>();
  return transB ? tc3_make<false, true>() : tc3_make<false, false>();
}

}  // namespace sg
