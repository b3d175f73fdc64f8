"""Single-precision GEMM for one NVIDIA GB300 (sm_103a).

    C = alpha * op(A) * op(B) + beta * C       (row-major FP32, op = N or T)

The computation happens entirely in the hand-written CUDA kernels of
``libsgemm_gb300.so`` (built from ``csrc/`` by ``build.py``); this package only
marshals arguments to its C ABI (``include/sgemm.h``) through ctypes.  PyTorch is
used for device memory and streams only.  There is no CPU fallback: every entry
point raises if the CUDA library is missing or cannot run.

Low level (same names and arguments as the C ABI, pointers as ints, raising
``SgemmError`` on any status other than success):
    sgemm, sgemm_ex, sgemm_strided_batched, sgemm_transpose, sgemm_noalloc,
    sgemm_select_algo, sgemm_last_launch_count,
    sgemm_last_device_status, sgemm_set_scratch_limit, sgemm_get_scratch_limit,
    sgemm_set_wait_budget_ns,
    sgemm_selftest_wait_timeout, sgemm_status_string, sgemm_algo_name,
    sgemm_version
High level (torch tensors): ``gemm``, ``gemm_strided_batched``, ``transpose``.
"""
from ._binding import (  # noqa: F401
    ALGO_AUTO, ALGO_NAIVE, ALGO_REG_2X2, ALGO_REG_4X4, ALGO_SIMT_CPASYNC, ALGO_SIMT_TMA,
    ALGO_SMALL, ALGO_SMEM_TILED, ALGO_TC_3XTF32,
    ALGOS, OP_N, OP_T, SCRATCH_UNLIMITED, STATUS, SgemmError, gemm, library_path, load_library,
    sgemm, sgemm_get_scratch_limit, sgemm_set_scratch_limit,
    sgemm_algo_name, sgemm_ex, sgemm_last_device_status, sgemm_last_launch_count, sgemm_noalloc,
    sgemm_select_algo, sgemm_selftest_wait_timeout, sgemm_set_wait_budget_ns,
    sgemm_status_string, sgemm_strided_batched, sgemm_transpose, sgemm_version,
    gemm_strided_batched, transpose)
