// Instantiations of the CUDA-core GEMM kernel: producer cpasync, op(A) = T.
#include "simt_instances.cuh"

namespace sg {
SG_DEFINE_SIMT_FAMILY(kCpAsync, 1)
}  // namespace sg
