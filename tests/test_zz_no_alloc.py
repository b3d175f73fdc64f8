"""sgemm_noalloc: the product for callers that may not let a library allocate
device memory -- programs whose own pool or caching allocator owns the GPU
memory (a cudaMalloc behind its back can fail or shrink the pool), loops that
cannot afford a cudaMalloc (it may synchronise the device and can fail under
memory pressure), and services whose memory footprint is fixed up front.

The entry point keeps its stream-K scratch in a fixed __device__ array instead
of a cudaMalloc'd workspace.  These tests call it through the C ABI and check,
on two calls in a row, that it gives what sgemm() gives and what the CPU oracle
gives (within the parity tolerance), including shapes whose split tiles go
through the scratch array; that its one-time set-up (the first call on a
device, an empty one included) is the only point where device memory is
reserved, in a fresh process; and that calls after it leave free device memory
unchanged.

This file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 20 * 1024 * 1024   # SGEMM_NOALLOC_SCRATCH_BYTES, include/sgemm.h

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
def test_noalloc_matches_sgemm_and_oracle_on_two_calls_in_a_row(orc, case):
    M, N, K, ta, tb, alpha, beta = case
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.rand((K, M) if ta else (M, K), generator=g).mul_(2).sub_(1).cuda()
    B = torch.rand((N, K) if tb else (K, N), generator=g).mul_(2).sub_(1).cuda()
    C0 = torch.rand((M, N), generator=g).mul_(2).sub_(1).cuda()

    ref = C0.clone()
    _call(sg.sgemm, ta, tb, M, N, K, alpha, A, B, beta, ref)
    torch.cuda.synchronize()
    R = orc.sgemm_f64(ta, tb, alpha, A.cpu().numpy(), B.cpu().numpy(), beta, C0.cpu().numpy())
    for call in range(2):
        out = C0.clone()
        _call(sg.sgemm_noalloc, ta, tb, M, N, K, alpha, A, B, beta, out)
        torch.cuda.synchronize()
        G = out.cpu().numpy()
        assert_close(G, ref.cpu().numpy().astype(np.float64), K,
                     f"noalloc call {call + 1} {M}x{N}x{K} against sgemm")
        assert_close(G, R, K, f"noalloc call {call + 1} {M}x{N}x{K} against the oracle")
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


def _setup_call():
    """An empty product (M = 0): only the one-time set-up of the device."""
    sg.sgemm_noalloc(0, 0, 0, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8,
                     torch.cuda.current_stream().cuda_stream)


def test_noalloc_uses_the_scratch_path_and_allocates_nothing():
    """After the set-up call, split (two-launch) products through
    sgemm_noalloc, repeated on new shapes and every op pair, leave the
    device's free memory exactly where it was."""
    shapes = [(2048, 2048, 2048), (1024, 1024, 1024), (3000, 2000, 1500)]
    bufs = []
    for (M, N, K) in shapes:
        bufs.append((torch.randn(M, K, device="cuda"), torch.randn(K, N, device="cuda"),
                     torch.empty(M, N, device="cuda")))
    torch.cuda.synchronize()
    _setup_call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for (M, N, K), (A, B, C) in zip(shapes, bufs):
        for _ in range(2):
            _call(sg.sgemm_noalloc, 0, 0, M, N, K, 1.0, A, B, 0.0, C)
            assert sg.sgemm_last_launch_count() == 2   # main kernel + fixup: scratch in use
    M = N = K = 1024   # square, so every op pair reads the same buffers
    A, B, C = bufs[1]
    for ta in (0, 1):
        for tb in (0, 1):
            _call(sg.sgemm_noalloc, ta, tb, M, N, K, 1.0, A, B, 0.5, C)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


_FRESH = r"""
import json, sys
import torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_matrix_10_gb300 as sg
torch.zeros(1, device="cuda")
A = torch.randn(2048, 2048, device="cuda")
B = torch.randn(2048, 2048, device="cuda")
C = torch.empty(2048, 2048, device="cuda")
torch.cuda.synchronize()
s = torch.cuda.current_stream().cuda_stream
f0 = torch.cuda.mem_get_info()[0]
sg.sgemm_noalloc(0, 0, 0, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8, s)   # set-up only
torch.cuda.synchronize()
f1 = torch.cuda.mem_get_info()[0]
for ta in (0, 1):
    for tb in (0, 1):
        # the offset of 4 bytes makes A and B misaligned: the cp.async producer
        for (M, N, K, off) in ((2048, 2048, 2048, 0), (1000, 1013, 997, 0), (1000, 1013, 997, 4),
                               (2048, 64, 2048, 0)):
            sg.sgemm_noalloc(ta, tb, M, N, K, 1.0, A.data_ptr() + off, 2048, B.data_ptr() + off,
                             2048, 0.5, C.data_ptr(), 2048, s)
torch.cuda.synchronize()
f2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"setup": f0 - f1, "calls": f1 - f2}))
"""


def test_setup_is_the_only_reservation_in_a_fresh_process(tmp_path):
    """In a process that has never called the library, the set-up call may
    reserve device memory (the scratch array and the kernels' code, loaded
    lazily by the CUDA runtime), at most the array plus a few MiB; the sixteen
    products that follow -- every op pair, TMA and cp.async producers, split
    and whole tiles -- reserve nothing more."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "fresh.py"
    script.write_text(_FRESH)
    out = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    got = json.loads(out.stdout.strip().splitlines()[-1])
    assert got["calls"] == 0, got
    assert 0 <= got["setup"] <= NOALLOC_SCRATCH_BYTES + (32 << 20), got


def test_noalloc_rejects_bad_arguments_like_sgemm():
    A = torch.randn(8, 8, device="cuda")
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_noalloc(0, 0, 8, 8, 8, 1.0, A.data_ptr(), 7, A.data_ptr(), 8, 0.0,
                         torch.empty(8, 8, device="cuda").data_ptr(), 8)
    assert e.value.status == 1
    assert "scratch" in sg.sgemm_status_string(6)
