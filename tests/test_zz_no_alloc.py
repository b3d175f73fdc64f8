"""sgemm_noalloc: the product for callers that may not let a library allocate
device memory (programs whose own allocator owns the GPU memory, loops that
cannot afford a synchronising cudaMalloc, fixed-footprint services).

The entry point keeps its stream-K scratch in a fixed array loaded with the
library instead of a cudaMalloc'd workspace.  These tests call it through the
C ABI and check, on two calls in a row, that it gives what sgemm() gives
(within the parity tolerance), including shapes whose split tiles go through
the scratch array, and that the calls leave free device memory unchanged.

This file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

# (M, N, K, transA, transB, alpha, beta): stream-K with scratch (2048^3 NN and
# TN, 1024^3, the 8192 x 64 x 4096 skinny product) and one that needs none.
CASES = [(2048, 2048, 2048, 0, 0, 1.0, 0.0), (1024, 1024, 1024, 1, 0, 1.5, 0.5),
         (8192, 64, 4096, 0, 0, 1.0, 1.0), (1000, 1013, 997, 0, 1, -1.0, 2.0),
         (152 * 128, 128, 256, 0, 0, 1.0, 0.0)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()


def _ptr_ld(t):
    return t.data_ptr(), (t.stride(0) if t.shape[0] > 1 else t.shape[1])


def _call(fn, ta, tb, M, N, K, alpha, A, B, beta, C):
    pa, lda = _ptr_ld(A)
    pb, ldb = _ptr_ld(B)
    pc, ldc = _ptr_ld(C)
    fn(ta, tb, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc,
       torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_{'NT'[c[3]]}{'NT'[c[4]]}" for c in CASES])
def test_noalloc_matches_sgemm_on_two_calls_in_a_row(case):
    M, N, K, ta, tb, alpha, beta = case
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.rand((K, M) if ta else (M, K), generator=g).mul_(2).sub_(1).cuda()
    B = torch.rand((N, K) if tb else (K, N), generator=g).mul_(2).sub_(1).cuda()
    C0 = torch.rand((M, N), generator=g).mul_(2).sub_(1).cuda()

    ref = C0.clone()
    _call(sg.sgemm, ta, tb, M, N, K, alpha, A, B, beta, ref)
    torch.cuda.synchronize()
    for call in range(2):
        out = C0.clone()
        _call(sg.sgemm_noalloc, ta, tb, M, N, K, alpha, A, B, beta, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), K,
                     f"noalloc call {call + 1} {M}x{N}x{K}")
    assert sg.sgemm_last_device_status() == 0


# (M, N, K, transA, transB, alpha, beta): both entry points take the 128 x 128
# tile (A read m-contiguous) and the same stream-K split (every tile split,
# at most three segments each)
SAME_SPLIT = [(1536, 1024, 1024, 1, 0, 1.5, 0.5), (1280, 1280, 768, 1, 1, 1.0, 0.0)]


@pytest.mark.parametrize("case", SAME_SPLIT, ids=["1536x1024x1024_TN", "1280x1280x768_TT"])
def test_in_kernel_fixup_equals_fixup_launch(case):
    """sgemm finishes split tiles inside the product kernel (the last CTA to
    arrive adds the partials); sgemm_noalloc leaves them to sk_fixup_kernel.
    Both add the same partials in the same k order: equal bit for bit."""
    M, N, K, ta, tb, alpha, beta = case
    g = torch.Generator().manual_seed(7 + M)
    A = torch.randn((K, M) if ta else (M, K), generator=g).cuda()
    B = torch.randn((N, K) if tb else (K, N), generator=g).cuda()
    C0 = torch.randn((M, N), generator=g).cuda()
    ref = C0.clone()
    _call(sg.sgemm, ta, tb, M, N, K, alpha, A, B, beta, ref)
    assert sg.sgemm_last_launch_count() == 1
    out = C0.clone()
    _call(sg.sgemm_noalloc, ta, tb, M, N, K, alpha, A, B, beta, out)
    assert sg.sgemm_last_launch_count() == 2
    torch.cuda.synchronize()
    assert torch.equal(ref, out)
    assert sg.sgemm_last_device_status() == 0


def test_noalloc_uses_the_scratch_path_and_allocates_nothing():
    """A split (two-launch) product through sgemm_noalloc, repeated on new
    shapes, leaves the device's free memory exactly where it was."""
    shapes = [(2048, 2048, 2048), (1024, 1024, 1024), (3000, 2000, 1500)]
    bufs = []
    for (M, N, K) in shapes:
        bufs.append((torch.randn(M, K, device="cuda"), torch.randn(K, N, device="cuda"),
                     torch.empty(M, N, device="cuda")))
    torch.cuda.synchronize()
    # first call on this device performs the one-time set-up
    A, B, C = bufs[0]
    _call(sg.sgemm_noalloc, 0, 0, 2048, 2048, 2048, 1.0, A, B, 0.0, C)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for (M, N, K), (A, B, C) in zip(shapes, bufs):
        for _ in range(2):
            _call(sg.sgemm_noalloc, 0, 0, M, N, K, 1.0, A, B, 0.0, C)
            assert sg.sgemm_last_launch_count() == 2   # main kernel + fixup: scratch in use
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_bad_arguments_like_sgemm():
    A = torch.randn(8, 8, device="cuda")
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_noalloc(0, 0, 8, 8, 8, 1.0, A.data_ptr(), 7, A.data_ptr(), 8, 0.0,
                         torch.empty(8, 8, device="cuda").data_ptr(), 8)
    assert e.value.status == 1
    assert "scratch" in sg.sgemm_status_string(6)
