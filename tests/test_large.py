"""Products and transposes whose operands hold more than 2^31 elements: every
element offset (row * ld + column, for A, B, C and the transpose's input and
output) is formed in 64-bit arithmetic.  The data follow closed forms, so the
expected outputs of any sampled rows are exact integers computed on the host
from the same formulas (no copy of the multi-GiB operands), and the GPU
result must equal them bit for bit (integer-valued FP32 products and sums
below 2^24 are exact in any order).
"""
import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg

pytestmark = pytest.mark.gpu

CHUNK_ELEMS = 1 << 27   # elements generated per step on the device (1 GiB of int64)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()
    if torch.cuda.mem_get_info()[0] < (48 << 30):
        pytest.skip("needs 48 GiB of free device memory")
    yield
    torch.cuda.empty_cache()


def a_val(i, k):
    return (i * 7 + k * 3) % 13 - 6


def b_val(k, j):
    return (k * 5 + j * 11) % 9 - 4


def fill(rows, cols, f, transpose=False):
    """A rows x cols device matrix with element (r, c) = f(r, c), built in
    chunks of rows (stored transposed if asked: cols x rows)."""
    out = torch.empty((cols, rows) if transpose else (rows, cols), device="cuda")
    c = torch.arange(cols, device="cuda", dtype=torch.int64)[None, :]
    step = max(1, CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        r = torch.arange(r0, r1, device="cuda", dtype=torch.int64)[:, None]
        v = f(r, c).to(torch.float32)
        if transpose:
            out[:, r0:r1] = v.t()
        else:
            out[r0:r1] = v
        del v, r
    return out


def expected_rows(rows, K, N):
    """Exact C rows (alpha 1, beta 0) for the given row indices."""
    i = np.asarray(rows, dtype=np.int64)[:, None, None]
    k = np.arange(K, dtype=np.int64)[None, :, None]
    j = np.arange(N, dtype=np.int64)[None, None, :]
    return (a_val(i, k) * b_val(k, j)).sum(axis=1).astype(np.float32)


@pytest.mark.parametrize("ta", [0, 1], ids=["A_MxK", "A_KxM"])
def test_a_with_more_than_2_31_elements(ta):
    """op(A) of 2^21 + 37 rows and K = 1100: A holds 2.3 G elements (stored
    M x K or K x M); N = 64 takes the skinny tile and stream-K."""
    M, K, N = (1 << 21) + 37, 1100, 64
    assert M * K > (1 << 31)
    A = fill(M, K, a_val, transpose=bool(ta))
    B = fill(K, N, b_val)
    C = torch.empty(M, N, device="cuda")
    sg.gemm(A, B, C, 1.0, 0.0, ta, 0)
    torch.cuda.synchronize()
    assert sg.sgemm_last_device_status() == 0
    rng = np.random.default_rng(7 + ta)
    rows = np.unique(np.concatenate([
        np.arange(M - 40, M),                                 # the last rows (offsets past 2^31)
        np.arange((1 << 31) // K - 20, (1 << 31) // K + 20),  # around element offset 2^31
        np.arange(0, 20), rng.integers(0, M, 60)]))
    G = C[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    np.testing.assert_array_equal(G, expected_rows(rows, K, N))
    del A, B, C


def test_c_with_more_than_2_31_elements():
    """C of 40000 x 60000 (2.4 G elements), K = 8: the epilogue's row offsets
    pass 2^31 elements; alpha and beta applied to an integer C."""
    M, N, K = 40000, 60000, 8
    assert M * N > (1 << 31)
    A = fill(M, K, a_val)
    B = fill(K, N, b_val)
    C = fill(M, N, lambda r, c: (r + 2 * c) % 5 - 2)
    sg.gemm(A, B, C, 2.0, -1.0)
    torch.cuda.synchronize()
    assert sg.sgemm_last_device_status() == 0
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.arange(M - 8, M), np.arange((1 << 31) // N - 4,
                                                                    (1 << 31) // N + 4),
                                     rng.integers(0, M, 16)]))
    G = C[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    c0 = ((rows[:, None] + 2 * np.arange(N)[None, :]) % 5 - 2).astype(np.float32)
    np.testing.assert_array_equal(G, 2.0 * expected_rows(rows, K, N) - c0)
    del A, B, C


def test_transpose_with_more_than_2_31_elements():
    """A 48000 x 48000 transpose (2.3 G elements each way), bit for bit
    against the closed form at sampled rows of the output."""
    n = 48000
    assert n * n > (1 << 31)
    X = fill(n, n, lambda r, c: (r * 3 + c * 7) % 1021)
    Y = sg.transpose(X)
    torch.cuda.synchronize()
    del X
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([np.arange(n - 8, n), rng.integers(0, n, 24)]))
    G = Y[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    # Y[c][r] = X[r][c]
    want = ((np.arange(n)[None, :] * 3 + rows[:, None] * 7) % 1021).astype(np.float32)
    np.testing.assert_array_equal(G, want)
    del Y


def test_strided_batch_beyond_2_31_elements():
    """2000 products of 1100 x 1100 by a shared 1100 x 64 (stride 0): the
    batch of A holds 2.4 G elements, so the later products' offsets pass 2^31;
    sampled rows of the first, middle and last products, bit for bit."""
    bt, M, K, N = 2000, 1100, 1100, 64
    assert bt * M * K > (1 << 31)
    A = torch.empty(bt, M, K, device="cuda")
    c = torch.arange(K, device="cuda", dtype=torch.int64)[None, :]
    r = torch.arange(M, device="cuda", dtype=torch.int64)[:, None]
    for b in range(bt):   # product b: rows offset by b
        A[b] = a_val(r + b, c).to(torch.float32)
    B = fill(K, N, b_val).expand(bt, K, N)
    C = sg.gemm_strided_batched(A, B)
    torch.cuda.synchronize()
    assert sg.sgemm_last_device_status() == 0
    rows = np.array([0, 1, 517, M - 1])
    for b in (0, 1, bt // 2, (1 << 31) // (M * K), bt - 2, bt - 1):
        G = C[b][torch.as_tensor(rows, device="cuda")].cpu().numpy()
        np.testing.assert_array_equal(G, expected_rows(rows + b, K, N), err_msg=f"product {b}")
    del A, B, C
