// Instantiations of the CUDA-core GEMM kernel: producer cpasync, op(A) = N.
#include "simt_instances.cuh"

namespace sg {
SG_DEFINE_SIMT_FAMILY(kCpAsync, 0)
}  // namespace sg
