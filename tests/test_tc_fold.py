"""The folded form of the 3xTF32 CTA-pair kernel (build option SG_TC_FOLD=1):
a k-contiguous operand is not split ahead; the product kernel computes its
small parts in shared memory from the TMA tile of the operand itself, with
the split pass's arithmetic.  The default build splits every operand ahead.

The test builds that variant of the library and checks, in a child process
that loads it, that every op pair gives the same bits as the default build on
the same operands (ragged tiles, alpha and beta included), that the launch
count drops by one per k-contiguous operand, and that the device status word
stays clean.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (M, N, K, ta, tb, alpha, beta)
CASES = [(2048, 2560, 512, 0, 0, 1.0, 0.0), (2048, 2560, 512, 0, 1, 1.0, 0.0),
         (2048, 2560, 512, 1, 1, 1.0, 0.0), (2048, 2560, 512, 1, 0, 1.0, 0.0),
         (1600, 4000, 512, 0, 0, 1.5, -0.5), (1600, 4000, 512, 0, 1, 1.5, -0.5),
         (2000, 2504, 1004, 0, 1, 1.25, -0.5), (1664, 1664, 4000, 0, 1, 0.75, 0.5)]

CHILD = r"""
import sys
import torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_matrix_10_gb300 as sg
assert sg.library_path() == sys.argv[2], sg.library_path()
data = torch.load(sys.argv[3])
for (M, N, K, ta, tb, alpha, beta), A, B, C0, ref in data:
    C = C0.cuda()
    sg.gemm(A.cuda(), B.cuda(), C, alpha, beta, ta, tb, algo="tc_3xtf32")
    n = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    what = f"{M}x{N}x{K} {ta}{tb}"
    assert n == 1 + ta + (1 - tb), f"{what}: {n} launches"
    assert torch.equal(C.cpu(), ref), f"{what}: differs from the split-ahead build"
st = sg.sgemm_last_device_status()
assert st == 0, st
print("ok")
"""


def test_folded_pair_kernel_matches_split_ahead(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_10_gb300 as sg
    from dense_fp32_matrix_10_gb300 import build
    g = torch.Generator().manual_seed(404)
    data = []
    for (M, N, K, ta, tb, alpha, beta) in CASES:
        A = torch.randn((K, M) if ta else (M, K), generator=g)
        B = torch.randn((N, K) if tb else (K, N), generator=g)
        C0 = torch.rand(M, N, generator=g).mul_(2).sub_(1)
        C = C0.cuda()
        sg.gemm(A.cuda(), B.cuda(), C, alpha, beta, ta, tb, algo="tc_3xtf32")
        assert sg.sgemm_last_launch_count() == 3
        torch.cuda.synchronize()
        data.append(((M, N, K, ta, tb, alpha, beta), A, B, C0, C.cpu()))
    torch.save(data, tmp_path / "cases.pt")
    lib = build.build(defines=["SG_TC_FOLD=1"],
                      out=os.path.join(build.BUILD, "libsgemm_gb300_tc_fold.so"))
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    env = dict(os.environ, SGEMM_GB300_LIBRARY=lib)
    out = subprocess.run([sys.executable, str(script), ROOT, lib, str(tmp_path / "cases.pt")],
                         capture_output=True, text=True, timeout=900, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-3000:]
    assert out.stdout.strip().endswith("ok")
