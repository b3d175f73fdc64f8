// Instantiations of the CUDA-core GEMM kernel: producer tma, op(A) = T.
#include "simt_instances.cuh"

namespace sg {
SG_DEFINE_SIMT_FAMILY(kTma, 1)
}  // namespace sg
