// Instantiations and host launch wrappers of the 3xTF32 tensor-core kernel
// (one per op(A) / op(B) layout).
#include "internal.h"
#include "tc_3xtf32.cuh"

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

TcEntry tc3_entry(int transA, int transB) {
  // A stored M x K (transA = N) and B stored N x K (transB = T) are k-contiguous.
  if (transA == 0) return transB ? tc3_make<true, true>() : tc3_make<true, false>();
  return transB ? tc3_make<false, true>() : tc3_make<false, false>();
}

}  // namespace sg
