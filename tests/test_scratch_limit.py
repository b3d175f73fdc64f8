"""The scratch limit (sgemm_set_scratch_limit): with a limit of 0, sgemm(),
sgemm_ex() and sgemm_strided_batched() allocate no device memory -- the caller
owns all of it, and the library only its status word -- and every workload
still matches the CPU oracle; a lower limit frees what the library holds; the
SGEMM_SCRATCH_LIMIT environment variable sets the initial limit.  All calls go
through the C ABI."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg
from dense_fp32_matrix_10_gb300 import workloads as W
from tests.parity import assert_bit_exact, assert_close

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
    sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
    assert sg.sgemm_last_device_status() == 0


# (case, kernel family): every workload family, the tensor-core family on the
# headline and NT shapes (whose split-ahead forms need scratch: under limit 0
# they run the one-launch form that splits in the kernel), and the integer
# variant of the NT workload
LIMIT0_CASES = [(c, "auto") for c in W.ALL_CASES] + [(W.HEADLINE, "tc_3xtf32"),
                                                     (W.NT_4096, "tc_3xtf32"),
                                                     (W.NT_4096.as_int(), "auto")]


def test_limit_zero_allocates_nothing_and_matches_the_oracle(orc):
    """Every workload under limit 0: the device's free memory and the bytes the
    library holds do not move, large products run as one launch when the
    library holds nothing (no stream-K fixup pass, no operand copied ahead),
    and each whole output matches the oracle (bit for bit on integer
    inputs)."""
    host = [(case, algo, W.make_inputs(case)) for case, algo in LIMIT0_CASES]
    dev = [tuple(t.cuda() for t in inputs) for _, _, inputs in host]
    torch.cuda.synchronize()
    sg.sgemm_set_scratch_limit(0)
    # a first pass makes the CUDA runtime load every kernel these calls launch
    # (lazy module loading takes device memory for code at a kernel's first
    # launch); C is restored from the host afterwards
    for (case, algo, _), (dA, dB, dC) in zip(host, dev):
        sg.gemm(dA, dB, dC, case.alpha, case.beta, case.transA, case.transB, algo=algo)
    for (_, _, (A, B, C)), (_, _, dC) in zip(host, dev):
        dC.copy_(C)
    torch.cuda.synchronize()
    held0 = sg.sgemm_get_scratch_limit()[1]   # buffers captured graphs still hold
    free0, _ = torch.cuda.mem_get_info()
    launches = {}
    for (case, algo, _), (dA, dB, dC) in zip(host, dev):
        sg.gemm(dA, dB, dC, case.alpha, case.beta, case.transA, case.transB, algo=algo)
        launches[case.name + algo] = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    limit, held1 = sg.sgemm_get_scratch_limit()
    sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
    assert limit == 0
    assert free1 == free0
    assert held1 == held0
    if held0 == 0:
        # nothing held (no graph kept a buffer): no fixup pass, nothing copied
        # ahead; buffers a graph still holds may be used, since using them
        # allocates nothing
        assert launches[W.HEADLINE.name + "auto"] == 1
        assert launches[W.SQUARE_1024.name + "auto"] == 1
        assert launches[W.HEADLINE.name + "tc_3xtf32"] == 1
        assert launches[W.NT_4096.name + "tc_3xtf32"] == 1
    for (case, algo, (A, B, C)), (_, _, dC) in zip(host, dev):
        R = orc.sgemm_f64(case.transA, case.transB, case.alpha, A.numpy(), B.numpy(), case.beta,
                          C.numpy() if case.beta != 0 else None)
        G = dC.cpu().numpy()
        if case.dist == "int":
            assert_bit_exact(G, R, f"{case.name} {algo} at limit 0")
        else:
            assert_close(G, R, case.K, f"{case.name} {algo} at limit 0")


def test_limit_zero_strided_batch(orc):
    """A strided batch large enough to be split by stream-K runs whole tiles
    under limit 0 and still matches the oracle product by product."""
    bt, M, N, K = 6, 384, 320, 1000
    g = torch.Generator().manual_seed(5)
    A = (torch.rand(bt, M, K, generator=g) * 2 - 1)
    B = (torch.rand(bt, K, N, generator=g) * 2 - 1)
    C = (torch.rand(bt, M, N, generator=g) * 2 - 1)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    sg.sgemm_set_scratch_limit(0)
    sg.gemm_strided_batched(dA, dB, dC, 1.25, -0.5)   # loads the kernels (see above)
    dC.copy_(C)
    torch.cuda.synchronize()
    held0 = sg.sgemm_get_scratch_limit()[1]
    free0, _ = torch.cuda.mem_get_info()
    sg.gemm_strided_batched(dA, dB, dC, 1.25, -0.5)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    held1 = sg.sgemm_get_scratch_limit()[1]
    sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
    assert (free1, held1) == (free0, held0)
    G = dC.cpu().numpy()
    for b in range(bt):
        R = orc.sgemm_f64(0, 0, 1.25, A[b].numpy(), B[b].numpy(), -0.5, C[b].numpy())
        assert_close(G[b], R, K, f"batch {b} at limit 0")


def test_limit_below_the_operand_scratch(orc):
    """A limit that admits the stream-K workspace (~40 MB) but not the 64 MiB an
    operand transpose of the headline product needs: the library never holds
    more than the limit (or what graphs already held), and the result still
    matches the oracle."""
    case = W.HEADLINE
    A, B, C = W.make_inputs(case)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
    held_before = sg.sgemm_get_scratch_limit()[1]
    limit = 48 << 20
    sg.sgemm_set_scratch_limit(limit)
    sg.gemm(dA, dB, dC)
    torch.cuda.synchronize()
    held = sg.sgemm_get_scratch_limit()[1]
    sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
    assert held <= max(limit, held_before)
    R = orc.sgemm_f64(0, 0, 1.0, A.numpy(), B.numpy())
    assert_close(dC.cpu().numpy(), R, case.K, "headline at a 48 MiB limit")


_FRESH = r"""
import json, sys
import torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_matrix_10_gb300 as sg
n = 4096
A = torch.randn(n, n, device="cuda"); B = torch.randn(n, n, device="cuda")
C = torch.empty(n, n, device="cuda")
out = {"initial_limit": sg.sgemm_get_scratch_limit()[0]}
sg.gemm(A, B, C); torch.cuda.synchronize()
out["held_after_product"] = sg.sgemm_get_scratch_limit()[1]
f0 = torch.cuda.mem_get_info()[0]
sg.sgemm_set_scratch_limit(0)
f1 = torch.cuda.mem_get_info()[0]
out["held_after_limit0"] = sg.sgemm_get_scratch_limit()[1]
out["freed"] = f1 - f0
sg.gemm(A, B, C); torch.cuda.synchronize()
out["held_after_second_product"] = sg.sgemm_get_scratch_limit()[1]
out["launches"] = sg.sgemm_last_launch_count()
print(json.dumps(out))
"""


def _fresh(tmp_path, env_limit=None):
    script = tmp_path / "fresh_limit.py"
    script.write_text(_FRESH)
    env = dict(os.environ)
    env.pop("SGEMM_SCRATCH_LIMIT", None)
    if env_limit is not None:
        env["SGEMM_SCRATCH_LIMIT"] = str(env_limit)
    out = subprocess.run([sys.executable, str(script), ROOT], capture_output=True, text=True,
                         timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_lowering_the_limit_frees_what_the_library_holds(tmp_path):
    """In a fresh process (no graphs): the headline product takes scratch
    (the operand transpose and the stream-K workspace); setting the limit to 0
    frees all of it and the next product allocates nothing."""
    got = _fresh(tmp_path)
    assert got["initial_limit"] == (1 << 64) - 1
    assert got["held_after_product"] > 0
    assert got["held_after_limit0"] == 0
    assert got["freed"] >= got["held_after_product"]
    assert got["held_after_second_product"] == 0
    assert got["launches"] == 1


def test_environment_sets_the_initial_limit(tmp_path):
    got = _fresh(tmp_path, env_limit=0)
    assert got["initial_limit"] == 0
    assert got["held_after_product"] == 0
    assert got["launches"] == 1
