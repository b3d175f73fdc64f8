"""CPU oracle for C = alpha * op(A) * op(B) + beta * C (single precision GEMM).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check in
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.  The
GPU library never imports or calls it, and it shares no code with the GPU path.

The arithmetic lives in ``oracle_sgemm.c`` (plain C, FP64 accumulation in
ascending k; its header comment gives the definition it follows and the pages
it cites).  This module is only ctypes marshalling of numpy arrays.  The library also
holds the transpose (``oracle_transpose_f32``) that the GPU transpose kernel
is checked against.

Matrices are 2-D numpy float32 arrays in their *stored* (row-major) layout:
A is M x K (op N) or K x M (op T); B is K x N (op N) or N x K (op T); C is M x N.
A row stride larger than the row length (a padded leading dimension) is
honoured; the element stride must be 1.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_I64 = ctypes.c_int64
_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)
_I64P = ctypes.POINTER(ctypes.c_int64)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _op(t):
    if t in (0, 1):
        return int(t)
    if isinstance(t, str) and len(t) == 1 and t in "NnTt":
        return 0 if t in "Nn" else 1
    raise ValueError("op must be 0/1 or 'N'/'T'")


def _mat(x, name):
    """(pointer, ld) of a 2-D float32 array with unit element stride."""
    if not isinstance(x, np.ndarray) or x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 numpy array")
    if x.size == 0:
        return None, max(x.shape[1], 1)
    if x.shape[1] > 1 and x.strides[1] != 4:
        raise ValueError(f"{name} must have unit element stride")
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    if x.strides[0] % 4 or ld < x.shape[1]:
        raise ValueError(f"{name} has an unusable row stride")
    return x.ctypes.data_as(_F32P), ld


def _shapes(ta, tb, A, B):
    M = A.shape[1] if ta else A.shape[0]
    Ka = A.shape[0] if ta else A.shape[1]
    Kb = B.shape[1] if tb else B.shape[0]
    N = B.shape[0] if tb else B.shape[1]
    if Ka != Kb:
        raise ValueError(f"inner dimensions differ: {Ka} vs {Kb}")
    return M, N, Ka


class Oracle:
    """Bound to one build of the oracle library (the default one, or another
    build of the same source such as a test's planted-mistake copy)."""

    def __init__(self, libpath=None):
        lib = ctypes.CDLL(libpath or _build.build())
        lib.oracle_sgemm_f64.restype = ctypes.c_int
        lib.oracle_sgemm_f64.argtypes = [
            ctypes.c_int, ctypes.c_int, _I64, _I64, _I64,
            ctypes.c_float, _F32P, _I64, _F32P, _I64,
            ctypes.c_float, _F32P, _I64, _F64P, _I64, ctypes.c_int]
        lib.oracle_transpose_f32.restype = ctypes.c_int
        lib.oracle_transpose_f32.argtypes = [_I64, _I64, _F32P, _I64, _F32P, _I64]
        lib.oracle_sgemm_entries_f64.restype = ctypes.c_int
        lib.oracle_sgemm_entries_f64.argtypes = [
            ctypes.c_int, ctypes.c_int, _I64, _I64, _I64,
            ctypes.c_float, _F32P, _I64, _F32P, _I64,
            ctypes.c_float, _F32P, _I64, _I64, _I64P, _I64P, _F64P]
        self.lib = lib

    def sgemm_f64(self, transA, transB, alpha, A, B, beta=0.0, C=None, threads=None):
        """The M x N float64 result alpha*op(A)*op(B) + beta*C."""
        ta, tb = _op(transA), _op(transB)
        M, N, K = _shapes(ta, tb, A, B)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        if C is not None:
            if C.shape != (M, N):
                raise ValueError("C has the wrong shape")
            pc, ldc = _mat(C, "C")
        else:
            pc, ldc = None, max(N, 1)
        R = np.empty((M, N), dtype=np.float64)
        st = self.lib.oracle_sgemm_f64(
            ta, tb, M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
            R.ctypes.data_as(_F64P), max(N, 1), int(threads or default_threads()))
        if st != 0:
            raise ValueError(f"oracle_sgemm_f64 rejected its arguments (status {st})")
        return R

    def sgemm_f32(self, transA, transB, alpha, A, B, beta=0.0, C=None, threads=None):
        """The FP64 result rounded once to FP32 (round to nearest even)."""
        return self.sgemm_f64(transA, transB, alpha, A, B, beta, C, threads).astype(np.float32)

    def sgemm_strided_batched_f64(self, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb,
                                  strideB, beta, C, ldc, strideC, batch, threads=None):
        """(batch, M, N) float64: product b is alpha*op(A_b)*op(B_b) + beta*C_b,
        where X_b is the stored matrix that starts b*strideX elements into the
        flat float32 buffer X, with leading dimension ldX (the strided-batch
        layout of BLAS-style interfaces; a stride of 0 repeats one matrix).
        Each product is one call of the single-product oracle on that offset;
        C may be None when beta == 0."""
        ta, tb = _op(transA), _op(transB)
        flats = []
        for x, name in ((A, "A"), (B, "B"), (C, "C")):
            if x is None:
                flats.append(None)
                continue
            if not isinstance(x, np.ndarray) or x.dtype != np.float32 or x.ndim != 1 \
                    or (x.size and x.strides[0] != 4):
                raise TypeError(f"{name} must be a contiguous 1-D float32 numpy array")
            flats.append(x)
        A, B, C = flats
        need = [(A, lda, strideA, K if ta else M, M if ta else K, "A"),
                (B, ldb, strideB, N if tb else K, K if tb else N, "B")]
        if C is not None:
            need.append((C, ldc, strideC, M, N, "C"))
        for x, ld, stride, rows, cols, name in need:
            if stride < 0 or ld < max(cols, 1):
                raise ValueError(f"{name}: bad stride or leading dimension")
            if batch > 0 and rows > 0 and cols > 0 and \
                    (batch - 1) * stride + (rows - 1) * ld + cols > x.size:
                raise ValueError(f"{name} buffer is too small for the batch")
        R = np.empty((batch, M, N), dtype=np.float64)
        nth = int(threads or default_threads())
        for b in range(batch):
            pa = ctypes.cast(A.ctypes.data + 4 * b * strideA, _F32P) if A is not None and A.size else None
            pb = ctypes.cast(B.ctypes.data + 4 * b * strideB, _F32P) if B is not None and B.size else None
            pc = ctypes.cast(C.ctypes.data + 4 * b * strideC, _F32P) if C is not None and C.size else None
            st = self.lib.oracle_sgemm_f64(
                ta, tb, M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
                R[b].ctypes.data_as(_F64P), max(N, 1), nth)
            if st != 0:
                raise ValueError(f"oracle_sgemm_f64 rejected product {b} (status {st})")
        return R

    def transpose_f32(self, X, out=None):
        """X^T of a 2-D float32 array (cols x rows, float32).  With `out` (a
        float32 array of that shape, possibly a view with a longer row) the
        result is written there and only there."""
        rows, cols = X.shape
        px, ldx = _mat(X, "X")
        if out is None:
            out = np.empty((cols, rows), dtype=np.float32)
        if out.shape != (cols, rows):
            raise ValueError("out has the wrong shape")
        po, ldo = _mat(out, "out")
        st = self.lib.oracle_transpose_f32(rows, cols, px, ldx, po, ldo)
        if st != 0:
            raise ValueError(f"oracle_transpose_f32 rejected its arguments (status {st})")
        return out

    def sgemm_entries_f64(self, transA, transB, alpha, A, B, beta, C, I, J):
        """float64 values of the (I[e], J[e]) outputs of the same product."""
        ta, tb = _op(transA), _op(transB)
        M, N, K = _shapes(ta, tb, A, B)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        pc, ldc = _mat(C, "C") if C is not None else (None, max(N, 1))
        I = np.ascontiguousarray(I, dtype=np.int64)
        J = np.ascontiguousarray(J, dtype=np.int64)
        if I.shape != J.shape or I.ndim != 1:
            raise ValueError("I and J must be 1-D and of equal length")
        R = np.empty(I.shape, dtype=np.float64)
        st = self.lib.oracle_sgemm_entries_f64(
            ta, tb, M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
            I.size, I.ctypes.data_as(_I64P), J.ctypes.data_as(_I64P), R.ctypes.data_as(_F64P))
        if st != 0:
            raise ValueError(f"oracle_sgemm_entries_f64 rejected its arguments (status {st})")
        return R


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def sgemm_f64(*args, **kw):
    return default().sgemm_f64(*args, **kw)


def sgemm_f32(*args, **kw):
    return default().sgemm_f32(*args, **kw)


def sgemm_entries_f64(*args, **kw):
    return default().sgemm_entries_f64(*args, **kw)


def sgemm_strided_batched_f64(*args, **kw):
    return default().sgemm_strided_batched_f64(*args, **kw)


def transpose_f32(*args, **kw):
    return default().transpose_f32(*args, **kw)
