"""Products captured into CUDA graphs.

The library's stream-K workspace and transpose scratch are shared by every
call on a device.  Inside a capture the library allocates nothing and orders
its uses of those buffers through external event nodes, so graph launches
and eager calls on other streams can be mixed.  These tests replay graphs
interleaved with eager stream-K / transposing calls on another stream and
require every result to be bit-identical to the same product run alone (a
race on the shared buffers would corrupt partial sums), plus a capture made
before any workspace exists (fresh process).
"""
import os
import subprocess
import sys

import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sg.sgemm_last_device_status() == 0


def _operands(M, N, K, seed, ta=0, tb=0):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn((K, M) if ta else (M, K), generator=g).cuda()
    B = torch.randn((N, K) if tb else (K, N), generator=g).cuda()
    return A, B


def _alone(A, B, M, N, ta=0, tb=0):
    C = torch.empty(M, N, device="cuda")
    sg.gemm(A, B, C, transA=ta, transB=tb)
    torch.cuda.synchronize()
    return C.clone()


# 1280 x 1024 x 1024: 80 tiles of 128 x 128, too many for clusters of two on
# 152 SMs, so stream-K with its workspace; 768 x 768 x 512 (36 tiles of 16
# k-tiles): cluster split-K
@pytest.mark.parametrize("shape", [(1280, 1024, 1024), (768, 768, 512), (2048, 4864, 256),
                                   (1000, 1013, 997), (2048, 2048, 2048)],
                         ids=["stream_k_1280x1024x1024", "cluster_split_768x768x512",
                              "pretransposed_2048x4864x256", "repacked_1000x1013x997",
                              "in_kernel_fixup_2048"])
def test_graph_replays_interleaved_with_eager_calls(shape):
    M, N, K = shape
    A1, B1 = _operands(M, N, K, 1)
    A2, B2 = _operands(M, N, K, 2)
    ref1, ref2 = _alone(A1, B1, M, N), _alone(A2, B2, M, N)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, N, device="cuda")
    with torch.cuda.stream(s1):
        sg.gemm(A1, B1, C1, stream=s1)                 # buffers exist before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        for _ in range(3):
            sg.gemm(A1, B1, C1, stream=s1)
    for _ in range(5):
        C1.zero_()
        torch.cuda.synchronize()
        g.replay()
        with torch.cuda.stream(s2):
            for _ in range(2):
                sg.gemm(A2, B2, C2, stream=s2)         # same shared buffers, other stream
        torch.cuda.synchronize()
        assert torch.equal(C1, ref1)
        assert torch.equal(C2, ref2)


def test_batched_and_transpose_capture():
    s = torch.cuda.Stream()
    A = torch.randn(16, 256, 64, device="cuda")
    B = torch.randn(16, 64, 256, device="cuda")
    X = torch.randn(3000, 1000, device="cuda")
    refC = sg.gemm_strided_batched(A, B)
    refT = sg.transpose(X)
    torch.cuda.synchronize()
    C = torch.empty_like(refC)
    T = torch.empty_like(refT)
    with torch.cuda.stream(s):
        sg.gemm_strided_batched(A, B, C, stream=s)
        sg.transpose(X, T, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sg.gemm_strided_batched(A, B, C, stream=s)
        sg.transpose(X, T, stream=s)
    C.zero_()
    T.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C, refC) and torch.equal(T, refT)


def test_batch_with_op_b_copied_ahead_in_graph():
    """A dense NT batch of 1024-row products copies op(B) transposed into the
    library scratch before the product (two launches).  Captured after an
    eager call has sized the scratch, its replays, interleaved with eager
    batches of another shape on another stream that share the scratch, equal
    the batch run alone bit for bit."""
    g0 = torch.Generator().manual_seed(21)
    A1 = torch.randn(10, 1024, 64, generator=g0).cuda()
    B1 = torch.randn(10, 512, 64, generator=g0).cuda()
    A2 = torch.randn(12, 1152, 96, generator=g0).cuda()
    B2 = torch.randn(12, 512, 96, generator=g0).cuda()
    ref1 = sg.gemm_strided_batched(A1, B1, transB=True)
    assert sg.sgemm_last_launch_count() == 2
    ref2 = sg.gemm_strided_batched(A2, B2, transB=True)
    assert sg.sgemm_last_launch_count() == 2
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    C1 = torch.empty_like(ref1)
    C2 = torch.empty_like(ref2)
    with torch.cuda.stream(s1):
        sg.gemm_strided_batched(A1, B1, C1, transB=True, stream=s1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        sg.gemm_strided_batched(A1, B1, C1, transB=True, stream=s1)
        assert sg.sgemm_last_launch_count() == 2
    for _ in range(4):
        C1.zero_()
        torch.cuda.synchronize()
        g.replay()
        with torch.cuda.stream(s2):
            sg.gemm_strided_batched(A2, B2, C2, transB=True, stream=s2)
        torch.cuda.synchronize()
        assert torch.equal(C1, ref1)
        assert torch.equal(C2, ref2)


GROW_CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r})
import dense_fp32_matrix_10_gb300 as sg
def ops(M, N, K, seed):
    g0 = torch.Generator().manual_seed(seed)
    return torch.randn(M, K, generator=g0).cuda(), torch.randn(K, N, generator=g0).cuda()
# a transposed-ahead product (scratch of K x M floats), captured
A, B = ops(2048, 4864, 256, 1)
C = torch.empty(2048, 4864, device="cuda")
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    sg.gemm(A, B, C, stream=s)
    assert sg.sgemm_last_launch_count() >= 2          # transpose + product
torch.cuda.synchronize()
ref = C.clone()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    sg.gemm(A, B, C, stream=s)
# an eager product needing a larger scratch (A^T of 8192 x 4096 floats, 128 MiB,
# against the 64 MiB allocated so far): gets a new buffer (its transpose ahead
# still runs) and must not free the graph's
A2, B2 = ops(4096, 4096, 8192, 2)
C2 = sg.gemm(A2, B2)
assert sg.sgemm_last_launch_count() >= 2
torch.cuda.synchronize()
C.zero_()
g.replay()
torch.cuda.synchronize()
assert torch.equal(C, ref)
r2 = A2.double() @ B2.double()
assert ((C2.double() - r2).norm() / r2.norm()).item() < 1e-5
assert sg.sgemm_last_device_status() == 0
print("ok")
"""


def test_captured_scratch_is_never_moved():
    """After a capture used the transpose scratch, a larger product must not
    free it (the graph holds its address): the larger product takes a new
    buffer and runs correctly, and the graph still replays correctly."""
    p = subprocess.run([sys.executable, "-c", GROW_CHILD.format(root=ROOT)], capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-3000:]
    assert p.stdout.strip().endswith("ok")


CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r})
import dense_fp32_matrix_10_gb300 as sg
M, N, K = 1280, 1024, 1024   # stream-K (more tiles than clusters of two fit)
g0 = torch.Generator().manual_seed(3)
A = torch.randn(M, K, generator=g0).cuda(); B = torch.randn(K, N, generator=g0).cuda()
C = torch.empty(M, N, device="cuda")
s = torch.cuda.Stream()
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):          # first call of the process: no workspace yet
    sg.gemm(A, B, C, stream=s)
g.replay(); torch.cuda.synchronize()
inside = C.clone()
C2 = sg.gemm(A, B)                           # eager afterwards: allocates, splits by stream-K
torch.cuda.synchronize()
ref = (A.double() @ B.double())
for X in (inside, C2):
    err = ((X.double() - ref).norm() / ref.norm()).item()
    assert err < 1e-5, err
assert sg.sgemm_last_device_status() == 0
print("ok")
"""


def test_capture_before_any_workspace_exists():
    p = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-3000:]
    assert p.stdout.strip().endswith("ok")


def test_tensor_core_pairs_in_graph():
    """A split-ahead 3xTF32 product runs as three launches, the last a
    cluster launch of CTA pairs.  Captured in a graph (after one eager call
    has sized the scratch), its replays, interleaved with eager tensor-core
    calls of another shape on another stream that share the scratch, equal
    the product run alone bit for bit."""
    M, N, K = 2048, 2560, 512
    A1, B1 = _operands(M, N, K, 7)
    A2, B2 = _operands(2048, 4096, 512, 8)

    def alone(A, B, m, n):
        C = torch.empty(m, n, device="cuda")
        sg.gemm(A, B, C, algo="tc_3xtf32")
        assert sg.sgemm_last_launch_count() == 3
        torch.cuda.synchronize()
        return C.clone()

    ref1, ref2 = alone(A1, B1, M, N), alone(A2, B2, 2048, 4096)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(2048, 4096, device="cuda")
    with torch.cuda.stream(s1):
        sg.gemm(A1, B1, C1, algo="tc_3xtf32", stream=s1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        sg.gemm(A1, B1, C1, algo="tc_3xtf32", stream=s1)
        assert sg.sgemm_last_launch_count() == 3
    for _ in range(4):
        C1.zero_()
        torch.cuda.synchronize()
        g.replay()
        with torch.cuda.stream(s2):
            sg.gemm(A2, B2, C2, algo="tc_3xtf32", stream=s2)
        torch.cuda.synchronize()
        assert torch.equal(C1, ref1)
        assert torch.equal(C2, ref2)
