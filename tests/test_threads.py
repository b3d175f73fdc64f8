"""Calls from several host threads at once.

The C ABI is thread-safe: per-device state is initialised once, and the
shared stream-K workspace and transpose scratch are guarded by locks and
ordered across streams by events.  ctypes releases the GIL during the call,
so these threads really overlap inside the library.  Each thread runs its
own products on its own stream; every result must equal, bit for bit, the
same product run alone.
"""
import threading

import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sg.sgemm_last_device_status() == 0


# (M, N, K, transA, transB, algo): stream-K splits (finished by the fixup
# pass, and in-kernel), a transpose ahead, the 3xTF32 split ahead, and a
# transpose on every thread
JOBS = [(1024, 1024, 1024, 0, 0, "auto"), (2048, 4864, 256, 0, 0, "auto"),
        (2048, 2560, 512, 1, 1, "tc_3xtf32"), (1536, 1024, 768, 1, 0, "auto"),
        (2048, 2048, 1024, 1, 0, "auto")]


def _job_inputs(i):
    M, N, K, ta, tb, algo = JOBS[i]
    g = torch.Generator().manual_seed(40 + i)
    A = torch.randn((K, M) if ta else (M, K), generator=g).cuda()
    B = torch.randn((N, K) if tb else (K, N), generator=g).cuda()
    return A, B


def test_concurrent_threads_match_lone_runs():
    inputs = [_job_inputs(i) for i in range(len(JOBS))]
    refs = []
    for (M, N, K, ta, tb, algo), (A, B) in zip(JOBS, inputs):
        C = torch.empty(M, N, device="cuda")
        sg.gemm(A, B, C, transA=ta, transB=tb, algo=algo)
        torch.cuda.synchronize()
        refs.append(C.clone())
    X = torch.randn(3000, 1000, device="cuda")
    Xt = sg.transpose(X)
    torch.cuda.synchronize()
    Xt = Xt.clone()

    errors = []
    outs = [[None] * 6 for _ in JOBS]

    def worker(i):
        try:
            M, N, K, ta, tb, algo = JOBS[i]
            A, B = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for r in range(6):
                    C = torch.empty(M, N, device="cuda")
                    sg.gemm(A, B, C, transA=ta, transB=tb, algo=algo, stream=s)
                    T = sg.transpose(X, stream=s)
                    outs[i][r] = (C, T)
            s.synchronize()
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(JOBS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    torch.cuda.synchronize()
    assert not errors, errors
    for i, ref in enumerate(refs):
        for r in range(6):
            C, T = outs[i][r]
            assert torch.equal(C, ref), (JOBS[i], r)
            assert torch.equal(T, Xt), (JOBS[i], r)
