"""ctypes marshalling for the C ABI of libsgemm_gb300.so (see include/sgemm.h).

Nothing here computes: every function forwards its arguments to the library.
The library is loaded on first use; if it is absent the call raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# SGEMM_GB300_LIBRARY may name another build of the same sources (for example a
# build with different compile-time kernel options).
_LIB_PATH = os.environ.get("SGEMM_GB300_LIBRARY") or os.path.join(HERE, "libsgemm_gb300.so")

OP_N, OP_T = 0, 1
(ALGO_AUTO, ALGO_SIMT_TMA, ALGO_SIMT_CPASYNC, ALGO_TC_3XTF32, ALGO_NAIVE, ALGO_SMEM_TILED,
 ALGO_SMALL, ALGO_REG_2X2, ALGO_REG_4X4) = range(9)
ALGOS = {"auto": ALGO_AUTO, "simt_tma": ALGO_SIMT_TMA, "simt_cpasync": ALGO_SIMT_CPASYNC,
         "tc_3xtf32": ALGO_TC_3XTF32, "naive": ALGO_NAIVE, "smem_tiled": ALGO_SMEM_TILED,
         "small": ALGO_SMALL, "reg_2x2": ALGO_REG_2X2, "reg_4x4": ALGO_REG_4X4}
STATUS = {0: "SGEMM_SUCCESS", 1: "SGEMM_ERR_INVALID_VALUE", 2: "SGEMM_ERR_ALIASING",
          3: "SGEMM_ERR_UNSUPPORTED", 4: "SGEMM_ERR_LAUNCH", 5: "SGEMM_ERR_DEVICE_TIMEOUT",
          6: "SGEMM_ERR_SCRATCH_LIMIT", 7: "SGEMM_ERR_DEVICE_BOUNDS"}

_lib = None
_I64 = ctypes.c_int64
_VP = ctypes.c_void_p


class SgemmError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} "
                         f"({sgemm_status_string(self.status)})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libsgemm_gb300.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -m dense_fp32_matrix_10_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(_LIB_PATH)
    gemm_args = [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64, ctypes.c_float, _VP, _I64,
                 _VP, _I64, ctypes.c_float, _VP, _I64, _VP]
    lib.sgemm.argtypes = gemm_args
    lib.sgemm.restype = ctypes.c_int
    lib.sgemm_ex.argtypes = gemm_args + [ctypes.c_int]
    lib.sgemm_ex.restype = ctypes.c_int
    lib.sgemm_strided_batched.argtypes = [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64,
                                          ctypes.c_float, _VP, _I64, _I64, _VP, _I64, _I64,
                                          ctypes.c_float, _VP, _I64, _I64, _I64, _VP]
    lib.sgemm_strided_batched.restype = ctypes.c_int
    lib.sgemm_transpose.argtypes = [_I64, _I64, _VP, _I64, _VP, _I64, _VP]
    lib.sgemm_transpose.restype = ctypes.c_int
    lib.sgemm_noalloc.argtypes = gemm_args
    lib.sgemm_noalloc.restype = ctypes.c_int
    lib.sgemm_select_algo.argtypes = [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64, _VP, _I64,
                                      _VP, _I64, ctypes.c_float, ctypes.c_float, _VP, _I64]
    lib.sgemm_select_algo.restype = ctypes.c_int
    lib.sgemm_last_launch_count.argtypes = []
    lib.sgemm_last_launch_count.restype = ctypes.c_int
    lib.sgemm_last_device_status.argtypes = [_VP]
    lib.sgemm_last_device_status.restype = ctypes.c_int
    lib.sgemm_set_scratch_limit.argtypes = [ctypes.c_uint64]
    lib.sgemm_set_scratch_limit.restype = ctypes.c_int
    lib.sgemm_get_scratch_limit.argtypes = [ctypes.POINTER(ctypes.c_uint64),
                                            ctypes.POINTER(ctypes.c_uint64)]
    lib.sgemm_get_scratch_limit.restype = ctypes.c_int
    lib.sgemm_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    lib.sgemm_set_wait_budget_ns.restype = None
    lib.sgemm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _VP]
    lib.sgemm_selftest_wait_timeout.restype = ctypes.c_int
    lib.sgemm_status_string.argtypes = [ctypes.c_int]
    lib.sgemm_status_string.restype = ctypes.c_char_p
    lib.sgemm_algo_name.argtypes = [ctypes.c_int]
    lib.sgemm_algo_name.restype = ctypes.c_char_p
    lib.sgemm_version.argtypes = []
    lib.sgemm_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _op(t):
    if isinstance(t, bool):
        return int(t)
    if isinstance(t, str) and len(t) == 1:
        return ord(t)
    return int(t)


def _check(st, where):
    if st != 0:
        raise SgemmError(st, where)


def sgemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """C = alpha*op(A)*op(B) + beta*C on `stream`; A, B, C are device pointers (int)."""
    _check(load_library().sgemm(_op(transA), _op(transB), M, N, K, alpha, A, lda, B, ldb, beta,
                                C, ldc, stream), "sgemm")


def sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None,
             algo=ALGO_AUTO):
    """As sgemm with the kernel family forced (``algo`` int or name)."""
    algo = ALGOS[algo] if isinstance(algo, str) else int(algo)
    _check(load_library().sgemm_ex(_op(transA), _op(transB), M, N, K, alpha, A, lda, B, ldb,
                                   beta, C, ldc, stream, algo), "sgemm_ex")


def sgemm_strided_batched(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                          beta, C, ldc, strideC, batch, stream=None):
    """C_b = alpha*op(A_b)*op(B_b) + beta*C_b for b < batch (pointers as ints,
    strides in elements; 0 shares an operand across the batch)."""
    _check(load_library().sgemm_strided_batched(
        _op(transA), _op(transB), M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
        strideC, batch, stream), "sgemm_strided_batched")


def sgemm_transpose(rows, cols, inp, ld_in, out, ld_out, stream=None):
    """out (cols x rows) = in (rows x cols) transposed; pointers as ints."""
    _check(load_library().sgemm_transpose(rows, cols, inp, ld_in, out, ld_out, stream),
           "sgemm_transpose")


def sgemm_noalloc(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    """As sgemm, for callers that may not let the library allocate device
    memory: the scratch is a fixed __device__ array, reserved by the first
    call on a device (an empty call with M = 0 does only that set-up)."""
    _check(load_library().sgemm_noalloc(_op(transA), _op(transB), M, N, K, alpha, A, lda, B, ldb,
                                        beta, C, ldc, stream), "sgemm_noalloc")


def sgemm_select_algo(transA, transB, M, N, K, A, lda, B, ldb, alpha, beta, C, ldc) -> int:
    return load_library().sgemm_select_algo(_op(transA), _op(transB), M, N, K, A, lda, B, ldb,
                                            alpha, beta, C, ldc)


def sgemm_last_launch_count() -> int:
    return load_library().sgemm_last_launch_count()


def sgemm_last_device_status(stream=None) -> int:
    """Synchronise `stream`; return (and clear) the device status code."""
    return load_library().sgemm_last_device_status(stream)


SCRATCH_UNLIMITED = (1 << 64) - 1


def sgemm_set_scratch_limit(nbytes: int):
    """Cap the device memory the library may own on the current device
    (0: none; SCRATCH_UNLIMITED: no cap)."""
    _check(load_library().sgemm_set_scratch_limit(int(nbytes)), "sgemm_set_scratch_limit")


def sgemm_get_scratch_limit():
    """(limit, bytes held now) on the current device."""
    lim, held = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(load_library().sgemm_get_scratch_limit(ctypes.byref(lim), ctypes.byref(held)),
           "sgemm_get_scratch_limit")
    return lim.value, held.value


def sgemm_set_wait_budget_ns(budget_ns: int):
    load_library().sgemm_set_wait_budget_ns(int(budget_ns))


def sgemm_selftest_wait_timeout(budget_ns: int, stream=None):
    _check(load_library().sgemm_selftest_wait_timeout(int(budget_ns), stream),
           "sgemm_selftest_wait_timeout")


def sgemm_status_string(status: int) -> str:
    return load_library().sgemm_status_string(int(status)).decode()


def sgemm_algo_name(algo: int) -> str:
    return load_library().sgemm_algo_name(int(algo)).decode()


def sgemm_version() -> str:
    return load_library().sgemm_version().decode()


# ------------------------------------------------------------------ torch
def _batched(t, name):
    """(pointer, batch, rows, cols, ld, stride) of a 3-D float32 CUDA tensor whose
    last dimension is contiguous (stride(0) may be 0: one matrix shared)."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 3:
        raise TypeError(f"{name} must be a 3-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    b, rows, cols = t.shape
    if cols > 1 and t.stride(2) != 1:
        raise ValueError(f"{name} must have unit column stride")
    ld = t.stride(1) if (rows > 1 or t.stride(1) >= cols) else cols
    return t.data_ptr(), b, rows, cols, max(ld, 1), t.stride(0) if b > 1 else 0


def _matrix(t, name):
    """(pointer, rows, cols, ld) of a 2-D float32 CUDA tensor with unit column stride."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    rows, cols = t.shape
    st0, st1 = t.stride()
    if cols > 1 and st1 != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    ld = st0 if (rows > 1 or st0 >= cols) else cols
    if ld < cols:
        raise ValueError(f"{name} has overlapping rows")
    return t.data_ptr(), rows, cols, max(ld, 1)


def _current_raw_stream(device_index):
    """cudaStream_t (as int) of torch's current stream on `device_index`."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def transpose(X, out=None, stream=None):
    """X^T of a 2-D float32 CUDA tensor (unit column stride, any row stride)
    through sgemm_transpose; `out` (cols x rows, unit column stride) is
    allocated when not given."""
    import torch
    px, rows, cols, ldx = _matrix(X, "X")
    if out is None:
        out = torch.empty((cols, rows), dtype=torch.float32, device=X.device)
    po, orow, ocol, ldo = _matrix(out, "out")
    if (orow, ocol) != (cols, rows):
        raise ValueError(f"out must be {cols} x {rows}")
    s = stream if stream is not None else torch.cuda.current_stream(X.device)
    with torch.cuda.device(X.device):
        sgemm_transpose(rows, cols, px, ldx, po, ldo, s.cuda_stream)
    return out


def gemm_strided_batched(A, B, C=None, alpha=1.0, beta=0.0, transA=False, transB=False,
                         stream=None):
    """Batched C[b] = alpha * op(A[b]) @ op(B[b]) + beta * C[b] on 3-D torch CUDA
    tensors (a batch dimension of stride 0, e.g. from expand(), shares that
    operand).  If C is None a new (batch, M, N) tensor is allocated."""
    import torch
    pa, ba, ra, ca, lda, sa = _batched(A, "A")
    pb, bb, rb, cb, ldb, sb = _batched(B, "B")
    batch = max(ba, bb)
    if ba not in (1, batch) or bb not in (1, batch):
        raise ValueError("batch sizes differ")
    M, Ka = (ca, ra) if transA else (ra, ca)
    Kb, N = (cb, rb) if transB else (rb, cb)
    if Ka != Kb:
        raise ValueError(f"inner dimensions differ: {Ka} vs {Kb}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((batch, M, N), dtype=torch.float32, device=A.device)
    pc, bc, rc, cc, ldc, sc = _batched(C, "C")
    if (bc, rc, cc) != (batch, M, N):
        raise ValueError(f"C must be {batch} x {M} x {N}")
    s = stream if stream is not None else torch.cuda.current_stream(A.device)
    with torch.cuda.device(A.device):
        sgemm_strided_batched(int(bool(transA)), int(bool(transB)), M, N, Ka, float(alpha), pa, lda,
                              sa if ba > 1 else 0, pb, ldb, sb if bb > 1 else 0, float(beta), pc,
                              ldc, sc, batch, s.cuda_stream)
    return C


def gemm(A, B, C=None, alpha=1.0, beta=0.0, transA=False, transB=False, algo=ALGO_AUTO,
         stream=None):
    """C = alpha * op(A) @ op(B) + beta * C with torch CUDA tensors (row-major views).

    A, B are in stored layout (A is K x M when transA, B is N x K when transB).
    If C is None a new M x N tensor is allocated (beta must then be 0).
    Runs on ``stream`` (a torch.cuda.Stream) or the current torch stream.
    """
    import torch
    pa, ra, ca, lda = _matrix(A, "A")
    pb, rb, cb, ldb = _matrix(B, "B")
    M, Ka = (ca, ra) if transA else (ra, ca)
    Kb, N = (cb, rb) if transB else (rb, cb)
    if Ka != Kb:
        raise ValueError(f"inner dimensions differ: {Ka} vs {Kb}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    pc, rc, cc, ldc = _matrix(C, "C")
    if (rc, cc) != (M, N):
        raise ValueError(f"C must be {M} x {N}")
    algo = ALGOS[algo] if isinstance(algo, str) else int(algo)
    dev = A.get_device()
    if dev == torch.cuda.current_device():
        s = stream.cuda_stream if stream is not None else _current_raw_stream(dev)
        st = (_lib or load_library()).sgemm_ex(1 if transA else 0, 1 if transB else 0, M, N, Ka,
                                               alpha, pa, lda, pb, ldb, beta, pc, ldc, s, algo)
        if st != 0:
            raise SgemmError(st, "sgemm_ex")
        return C
    s = stream if stream is not None else torch.cuda.current_stream(A.device)
    with torch.cuda.device(A.device):
        sgemm_ex(int(bool(transA)), int(bool(transB)), M, N, Ka, float(alpha), pa, lda, pb, ldb,
                 float(beta), pc, ldc, s.cuda_stream, algo)
    return C
