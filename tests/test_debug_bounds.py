"""The debug-bounds build (SGEMM_DEBUG_BOUNDS=1): the kernels check the shared-
and global-memory indices they form and record SGEMM_ERR_DEVICE_BOUNDS in the
device status word instead of making an out-of-range access.  compute-sanitizer
is not available on this GPU pool; this build, the guard-band tests and the
comparisons with the oracle stand in for it.

The test builds that variant of the library and runs, in a child process that
loads it, tiny and tile-edge shapes over every kernel family and op pair, the
split forms (stream-K with the fixup pass and in-kernel, cluster split-K),
operands copied ahead (transposed, repacked), a strided batch and the
transpose -- each result against the CPU oracle, and the status word clean
after every group.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_matrix_10_gb300 as sg
import oracle
from tests.parity import assert_close

orc = oracle.default()
assert sg.library_path() == sys.argv[2], sg.library_path()
g = torch.Generator().manual_seed(99)

def rnd(*shape):
    return (torch.rand(*shape, generator=g) * 2 - 1)

def padded(X, tma):
    # a NaN-padded copy; rows of 16-byte multiples (plus one spare float4)
    # for the TMA families, one spare float otherwise
    pad = (-X.shape[1]) % 4 + 4 if tma else 1
    d = torch.full((X.shape[0], X.shape[1] + pad), float("nan"), device="cuda")[:, :X.shape[1]]
    d.copy_(X)
    return d

def product(M, N, K, ta, tb, algo, alpha=1.25, beta=-0.5):
    A = rnd(*((K, M) if ta else (M, K))); B = rnd(*((N, K) if tb else (K, N))); C = rnd(M, N)
    tma = algo in ("simt_tma", "tc_3xtf32")
    dA, dB = padded(A, tma), padded(B, tma)
    dC = C.cuda()
    sg.gemm(dA, dB, dC, alpha, beta, ta, tb, algo=algo)
    torch.cuda.synchronize()
    R = orc.sgemm_f64(ta, tb, alpha, A.numpy(), B.numpy(), beta, C.numpy())
    assert_close(dC.cpu().numpy(), R, K, f"{algo} {M}x{N}x{K} {ta}{tb}")

def status(what):
    st = sg.sgemm_last_device_status()
    assert st == 0, f"{what}: device status {st} ({sg.sgemm_status_string(st)})"

tiny = [(1, 1, 1), (3, 5, 7), (7, 2, 6), (33, 31, 29), (129, 65, 33), (128, 128, 32), (127, 257, 97)]
for algo in ["simt_tma", "simt_cpasync", "small", "naive", "smem_tiled", "reg_2x2", "reg_4x4", "tc_3xtf32"]:
    for (M, N, K) in tiny:
        for ta in (0, 1):
            for tb in (0, 1):
                product(M, N, K, ta, tb, algo)
    status(algo)
# split forms and operands copied ahead, through AUTO
for (M, N, K, ta, tb) in [(512, 512, 512, 0, 0), (700, 650, 500, 0, 1), (1280, 1024, 1024, 0, 0),
                          (1280, 1024, 1024, 1, 0), (2048, 2048, 1024, 0, 1), (1000, 1013, 997, 0, 0),
                          (8192, 64, 1024, 0, 0), (300, 260, 1000, 1, 1)]:
    product(M, N, K, ta, tb, "auto")
status("auto")
product(2048, 2560, 512, 0, 0, "tc_3xtf32")
status("tc_3xtf32 split ahead")
# strided batch and transpose
Q = rnd(6, 200, 64).cuda(); Kt = rnd(6, 300, 64).cuda()
S = sg.gemm_strided_batched(Q, Kt, transB=True)
torch.cuda.synchronize()
for b in range(6):
    R = orc.sgemm_f64(0, 1, 1.0, Q[b].cpu().numpy(), Kt[b].cpu().numpy())
    assert_close(S[b].cpu().numpy(), R, 64, f"batch {b}")
X = rnd(1000, 777).cuda()
assert torch.equal(sg.transpose(X), X.t())
X = rnd(1024, 4096).cuda()
assert torch.equal(sg.transpose(X), X.t())
status("batch and transpose")
print("ok")
"""


def test_debug_bounds_build_runs_clean(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    lib = build.build(defines=["SGEMM_DEBUG_BOUNDS=1"],
                      out=os.path.join(build.BUILD, "libsgemm_gb300_debug_bounds.so"))
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    env = dict(os.environ, SGEMM_GB300_LIBRARY=lib)
    out = subprocess.run([sys.executable, str(script), ROOT, lib], capture_output=True, text=True,
                         timeout=900, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-3000:]
    assert out.stdout.strip().endswith("ok")
