// Instantiations of the CUDA-core GEMM kernel: producer tma, op(A) = N.
#include "simt_instances.cuh"

namespace sg {
SG_DEFINE_SIMT_FAMILY(kTma, 0)
}  // namespace sg
