"""sgemm_strided_batched: many independent products in one call.

Host-side argument checks run without a GPU (fake addresses, nothing is
launched).  The GPU tests compare every product of a batch with the oracle's
strided-batch function, element by element: attention-shaped batches (many
heads of small Q K^T products, head-interleaved rows), ragged shapes over all
four op combinations, shared (stride 0) operands, padded and misaligned
strides (the cp.async producer), batches large enough for stream-K, integer
data bit-exact, and the degenerate cases.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg
from tests.parity import assert_bit_exact, assert_close

FAKE_A, FAKE_B, FAKE_C = 0x10000, 0x4000000, 0x8000000


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_10_gb300 import build
    return ctypes.CDLL(build.build())


def _raw(lib, ta, tb, M, N, K, A, lda, sa, B, ldb, sb, C, ldc, sc, batch, alpha=1.0, beta=0.0):
    f = lib.sgemm_strided_batched
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    return f(ta, tb, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C, ldc, sc, batch, None)


# ------------------------------------------------------------------ host only
def test_bad_batch_or_stride_is_invalid(lib):
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_C, 4, 16, -1) == 1
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, -16, FAKE_B, 4, 16, FAKE_C, 4, 16, 2) == 1
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_C, 4, -16, 2) == 1
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 3, 16, FAKE_B, 4, 16, FAKE_C, 4, 16, 2) == 1  # lda < K


def test_overlapping_outputs_are_aliasing(lib):
    # C_b of 4 x 4 with ldc 4 spans 16 elements: strideC 15 overlaps C_0 and C_1
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_C, 4, 15, 2) == 2
    # padded rows: span is (4-1)*8 + 4 = 28 elements
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_C, 8, 27, 3) == 2
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_C, 8, 28, 3) in (0, 3)


def test_outputs_meeting_inputs_across_the_batch_are_aliasing(lib):
    # A_b at FAKE_A + 64 b (16 floats each, batch 8 -> 512 bytes); C placed at A_5
    # batch 2 spans only A_0 .. A_1: no overlap
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_A + 5 * 64, 4, 16, 2) in (0, 3)
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_A + 5 * 64, 4, 16, 8) == 2
    # C after the last B_b is fine; C over a shared (stride 0) B is not
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 16, FAKE_B + 8 * 64, 4, 16, 8) in (0, 3)
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 16, FAKE_B, 4, 0, FAKE_B + 32, 4, 16, 8) == 2


def test_inputs_may_overlap_each_other(lib):
    # A and B in one buffer (sliding windows): allowed
    assert _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 4, FAKE_A + 16, 4, 4, FAKE_C, 4, 16, 8) in (0, 3)


def test_empty_batches_do_nothing(lib):
    assert _raw(lib, 0, 0, 4, 4, 4, 0, 4, 0, 0, 4, 0, 0, 4, 0, 0) == 0
    assert lib.sgemm_last_launch_count() == 0
    assert _raw(lib, 0, 0, 0, 4, 4, 0, 4, 0, 0, 4, 0, 0, 4, 0, 5) == 0
    assert lib.sgemm_last_launch_count() == 0


def test_huge_strides_do_not_overflow_the_checks(lib):
    # (batch - 1) * stride far beyond 2^63 bytes must not wrap into "no overlap"
    big = 1 << 40
    st = _raw(lib, 0, 0, 4, 4, 4, FAKE_A, 4, big, FAKE_B, 4, 16, FAKE_A + 64, 4, 16, 1 << 30)
    assert st == 2


# ------------------------------------------------------------------ GPU
gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sg.sgemm_last_device_status() == 0


def _flat(n, kind, g, fill=float("nan")):
    if kind == "int":
        return torch.randint(-8, 9, (n,), generator=g).float()
    if kind == "nan":
        return torch.full((n,), fill)
    return torch.rand((n,), generator=g).mul_(2).sub_(1)


def _layout(ta, tb, M, N, K, lda=None, ldb=None, ldc=None):
    ar, ac = (K, M) if ta else (M, K)
    br, bc = (N, K) if tb else (K, N)
    return (ar, ac, lda or ac), (br, bc, ldb or bc), (M, N, ldc or N)


def _span(rows, cols, ld):
    return (rows - 1) * ld + cols if rows > 0 and cols > 0 else 0


def run_batched(orc, ta, tb, M, N, K, batch, alpha=1.0, beta=0.0, kind="float", lda=None, ldb=None,
                ldc=None, sa=None, sb=None, sc=None, offs=(0, 0, 0), seed=0, check="close"):
    """Fill flat buffers (NaN outside the matrices), run the GPU batch, compare
    every product with the oracle, and check that no element outside the C_b
    was written.  Returns the GPU result (batch, M, N)."""
    (ar, ac, lda), (br, bc, ldb), (cr, cc, ldc) = _layout(ta, tb, M, N, K, lda, ldb, ldc)
    sa = _span(ar, ac, lda) if sa is None else sa
    sb = _span(br, bc, ldb) if sb is None else sb
    sc = _span(cr, cc, ldc) if sc is None else sc
    g = torch.Generator().manual_seed(seed)
    bufs = []
    for (rows, cols, ld, st, off) in ((ar, ac, lda, sa, offs[0]), (br, bc, ldb, sb, offs[1]),
                                      (cr, cc, ldc, sc, offs[2])):
        n = off + (batch - 1) * st + _span(rows, cols, ld) + 7
        f = _flat(n, "nan", g)
        for b in range(batch if st else 1):
            for r in range(rows):
                s0 = off + b * st + r * ld
                f[s0: s0 + cols] = _flat(cols, kind, g)
        bufs.append(f)
    hA, hB, hC = bufs
    if beta == 0.0:
        hC = hC.clone()   # C's matrices hold values but are never read
    dA, dB, dC = hA.cuda(), hB.cuda(), hC.cuda()
    sg.sgemm_strided_batched(ta, tb, M, N, K, alpha, dA.data_ptr() + 4 * offs[0], lda, sa,
                             dB.data_ptr() + 4 * offs[1], ldb, sb, beta,
                             dC.data_ptr() + 4 * offs[2], ldc, sc, batch,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = dC.cpu()
    R = orc.sgemm_strided_batched_f64(
        ta, tb, M, N, K, alpha, hA.numpy()[offs[0]:], lda, sa, hB.numpy()[offs[1]:], ldb, sb, beta,
        hC.numpy()[offs[2]:] if beta != 0.0 else None, ldc, sc, batch)
    # every element outside the C_b is untouched
    mask = torch.zeros_like(out, dtype=torch.bool)
    G = np.empty((batch, M, N), np.float32)
    for b in range(batch):
        for r in range(M):
            s0 = offs[2] + b * sc + r * ldc
            mask[s0: s0 + N] = True
            G[b, r] = out[s0: s0 + N].numpy()
    same = (out[~mask] == hC[~mask]) | (torch.isnan(out[~mask]) & torch.isnan(hC[~mask]))
    assert bool(torch.all(same)), "an element outside the outputs was written"
    for b in range(batch):
        if check == "exact":
            assert_bit_exact(G[b], R[b], f"product {b}")
        else:
            assert_close(G[b], R[b], K, f"product {b}")
    return G


ATTN = [  # (batch, M, N, K, ta, tb): per-head Q K^T (NT) and P V (NN) shapes
    (32, 128, 128, 64, 0, 1), (16, 256, 256, 64, 0, 1), (12, 197, 197, 64, 0, 1),
    (32, 128, 64, 128, 0, 0), (8, 77, 64, 77, 0, 0)]


@gpu
@pytest.mark.parametrize("case", ATTN, ids=[f"b{c[0]}_{c[1]}x{c[2]}x{c[3]}_{'NT'[c[4]]}{'NT'[c[5]]}"
                                            for c in ATTN])
def test_attention_shapes(_cuda, orc, case):
    batch, M, N, K, ta, tb = case
    run_batched(orc, ta, tb, M, N, K, batch, alpha=0.125, seed=batch + M)


@gpu
@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
def test_ragged_all_ops_with_beta(_cuda, orc, op):
    ta, tb = op
    run_batched(orc, ta, tb, 127, 129, 33, 5, alpha=1.5, beta=-0.5, seed=3)
    run_batched(orc, ta, tb, 130, 260, 200, 3, alpha=-1.0, beta=2.0, seed=4)


@gpu
@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
def test_integer_bit_exact(_cuda, orc, op):
    ta, tb = op
    run_batched(orc, ta, tb, 200, 136, 96, 6, alpha=1.0, beta=1.0, kind="int", seed=5, check="exact")


@gpu
def test_head_interleaved_rows(_cuda, orc):
    """Q and K with all heads in one row (lda = heads * d, strideA = d): the
    layout of a packed projection output."""
    heads, S, d = 8, 96, 64
    run_batched(orc, 0, 1, S, S, d, heads, lda=heads * d, sa=d, ldb=heads * d, sb=d, seed=6)


@gpu
def test_shared_operands(_cuda, orc):
    # one weight matrix for every product (strideB = 0), then one A for all
    run_batched(orc, 0, 0, 100, 96, 80, 7, sb=0, beta=1.0, seed=7)
    run_batched(orc, 0, 1, 64, 130, 72, 5, sa=0, seed=8)


@gpu
def test_padded_strides_and_gaps(_cuda, orc):
    # strides beyond the matrices' span (gaps hold NaN and must stay so)
    run_batched(orc, 0, 0, 96, 100, 64, 4, lda=68, ldb=104, ldc=108, sa=96 * 68 + 36,
                sb=64 * 104 + 12, sc=96 * 108 + 20, beta=0.5, seed=9)


@gpu
def test_misaligned_strides_use_cpasync(_cuda, orc):
    # odd strides / offsets: not 16-byte aligned, the cp.async producer
    run_batched(orc, 0, 0, 70, 90, 50, 5, sa=70 * 50 + 1, sb=50 * 90 + 3, sc=70 * 90 + 5, seed=10)
    run_batched(orc, 1, 1, 70, 90, 50, 3, offs=(1, 2, 3), beta=1.0, seed=11)


@gpu
def test_overlapping_inputs(_cuda, orc):
    """Inputs of consecutive products overlapping (stride smaller than a
    matrix): legal, and read through the cp.async producer."""
    run_batched(orc, 0, 0, 64, 64, 64, 6, sa=16 * 64, sb=8 * 64, seed=12)


@gpu
def test_staged_epilogue_batch_gaps(_cuda, orc):
    """128 x 128 tiles of a batch written by 3-D TMA stores (beta = 0): C_b
    ragged in M and N (N % 4 == 0), with NaN-filled gaps inside ldc and
    between the C_b that must stay untouched."""
    run_batched(orc, 1, 0, 300, 260, 128, 16, alpha=0.75, ldb=264, sb=128 * 264, ldc=268,
                sc=300 * 268 + 36, seed=21)
    run_batched(orc, 0, 0, 257, 132, 64, 72, ldb=132, sb=64 * 132, ldc=136, sc=257 * 136 + 8,
                seed=22)
    # N % 4 != 0: the register epilogue (exact at the row ends)
    run_batched(orc, 1, 0, 300, 261, 128, 16, alpha=0.75, ldb=264, sb=128 * 264, ldc=268,
                sc=300 * 268 + 36, seed=23)


@gpu
def test_stream_k_batch(_cuda, orc):
    """A batch whose tiles outnumber the SMs once but not twice: the k-loop
    of the last wave is split and summed by the fixup pass."""
    G = run_batched(orc, 0, 0, 512, 512, 1024, 12, seed=13)
    assert sg.sgemm_last_launch_count() == 2
    G2 = run_batched(orc, 0, 0, 512, 512, 1024, 12, seed=13)
    assert np.array_equal(G, G2), "stream-K batch is not deterministic"
    run_batched(orc, 1, 0, 384, 640, 768, 10, kind="int", seed=14, check="exact")


@gpu
def test_wide_tile_batch(_cuda, orc):
    """Batches whose 128 x 256 tiles fill a wave run them: NN (A transposed in
    shared memory by the producer warps) and TN, ragged M, alpha and beta
    (staged TMA stores and the register epilogue), integer data exact."""
    run_batched(orc, 0, 0, 200, 512, 80, 40, seed=31)
    run_batched(orc, 1, 0, 200, 512, 80, 40, alpha=0.5, beta=-1.5, seed=32)
    run_batched(orc, 0, 0, 130, 256, 64, 80, kind="int", seed=33, check="exact")


@gpu
def test_nt_batch_with_op_b_transposed_ahead(_cuda, orc):
    """A batch of k-contiguous op(B) in dense consecutive blocks, products of
    1024 rows: op(B) is transposed once for the whole batch (two launches)
    and the batch runs the 128 x 256 tile; every product against the oracle,
    with alpha and beta, and integer data bit-exact.  Padded leading
    dimensions (not dense blocks) keep the one-launch path."""
    run_batched(orc, 0, 1, 1024, 512, 64, 10, alpha=1.5, beta=-0.5, seed=41)
    assert sg.sgemm_last_launch_count() == 2
    run_batched(orc, 0, 1, 1030, 512, 96, 10, kind="int", seed=42, check="exact")
    assert sg.sgemm_last_launch_count() == 2
    run_batched(orc, 0, 1, 1024, 512, 64, 10, ldb=68, seed=43)
    assert sg.sgemm_last_launch_count() == 1


@gpu
def test_single_product_matches_sgemm(_cuda):
    M, N, K = 300, 200, 152   # 16-byte rows: both calls take the TMA kernel
    A = torch.randn(M, K, device="cuda")
    B = torch.randn(K, N, device="cuda")
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, N, device="cuda")
    sg.gemm(A, B, C1, algo="simt_tma")
    sg.gemm_strided_batched(A[None], B[None], C2[None])
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


@gpu
def test_degenerate(_cuda):
    M, N, batch = 33, 47, 4
    C0 = torch.rand(batch, M, N, device="cuda")
    nanA = torch.full((batch, M, 8), float("nan"), device="cuda")
    nanB = torch.full((batch, 8, N), float("nan"), device="cuda")
    C = C0.clone()
    sg.gemm_strided_batched(nanA, nanB, C, alpha=0.0, beta=2.0)     # alpha == 0: C = beta * C
    torch.cuda.synchronize()
    assert torch.equal(C, 2.0 * C0)
    C = torch.full((batch, M, N), float("nan"), device="cuda")
    sg.gemm_strided_batched(torch.empty(batch, M, 0, device="cuda"),
                            torch.empty(batch, 0, N, device="cuda"), C)   # K == 0, beta == 0
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))
    assert sg.sgemm_last_launch_count() == 1


@gpu
def test_beta_zero_ignores_nan_in_c(_cuda, orc):
    batch, M, N, K = 3, 50, 60, 40
    A = torch.rand(batch, M, K, device="cuda")
    B = torch.rand(batch, K, N, device="cuda")
    C = torch.full((batch, M, N), float("nan"), device="cuda")
    sg.gemm_strided_batched(A, B, C)
    torch.cuda.synchronize()
    for b in range(batch):
        R = orc.sgemm_f64(0, 0, 1.0, A[b].cpu().numpy(), B[b].cpu().numpy())
        assert_close(C[b].cpu().numpy(), R, K, f"product {b}")


@gpu
def test_torch_wrapper_broadcast(_cuda, orc):
    """gemm_strided_batched with an expand()ed operand (batch stride 0)."""
    batch, M, N, K = 6, 80, 72, 48
    A = torch.rand(batch, M, K, device="cuda")
    W = torch.rand(1, N, K, device="cuda")
    C = sg.gemm_strided_batched(A, W.expand(batch, N, K), transB=True, alpha=2.0)
    torch.cuda.synchronize()
    for b in range(batch):
        R = orc.sgemm_f64(0, 1, 2.0, A[b].cpu().numpy(), W[0].cpu().numpy())
        assert_close(C[b].cpu().numpy(), R, K, f"product {b}")


@gpu
def test_stream_is_respected(_cuda, orc):
    s = torch.cuda.Stream()
    batch, M, N, K = 4, 256, 256, 256
    A = torch.rand(batch, M, K, device="cuda")
    B = torch.rand(batch, K, N, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = sg.gemm_strided_batched(A, B, stream=s)
    s.synchronize()
    for b in (0, batch - 1):
        R = orc.sgemm_f64(0, 0, 1.0, A[b].cpu().numpy(), B[b].cpu().numpy())
        assert_close(C[b].cpu().numpy(), R, K, f"product {b}")
