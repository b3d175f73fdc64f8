"""GPU results of the C ABI against the CPU oracle, element by element.

Covers every workload family (every output compared, at the full sizes too,
with random and with integer-valued inputs, the latter bit for bit), the
four op combinations through every kernel family, ragged tails spanning
several tiles, padded and misaligned leading dimensions, and the degenerate
cases.  All calls go through the C ABI (ctypes binding).
"""
import math

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg
from dense_fp32_matrix_10_gb300 import workloads as W
from tests.parity import (assert_bit_exact, assert_close, offset_view, padded, sample_indices)

pytestmark = pytest.mark.gpu

OPS = [(0, 0), (0, 1), (1, 0), (1, 1)]
GEMM_ALGOS = ["simt_tma", "simt_cpasync", "tc_3xtf32", "small", "reg_2x2", "reg_4x4"]
ANY_LAYOUT_ALGOS = ("simt_cpasync", "small", "reg_2x2", "reg_4x4")   # any alignment and ld
ALL_ALGOS = ["auto", "simt_tma", "simt_cpasync", "tc_3xtf32", "naive", "smem_tiled", "small",
             "reg_2x2", "reg_4x4"]
TMA_ALGOS = ("simt_tma", "tc_3xtf32")   # need 16-byte aligned rows


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sg.sgemm_last_device_status() == 0


def run_case(case, algo="auto", A=None, B=None, C=None):
    """Run `case` on the GPU; returns (GPU result, host inputs).  Forced TMA
    runs get leading dimensions padded up to a multiple of 4 (16-byte rows)."""
    if A is None:
        A, B, C = W.make_inputs(case)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    if algo in TMA_ALGOS:
        dA = padded(dA, (-A.shape[1]) % 4)
        dB = padded(dB, (-B.shape[1]) % 4)
    sg.gemm(dA, dB, dC, case.alpha, case.beta, case.transA, case.transB, algo=algo)
    torch.cuda.synchronize()
    return dC.cpu().numpy(), (A.numpy(), B.numpy(), C.numpy())


def oracle_full(orc, case, A, B, C):
    return orc.sgemm_f64(case.transA, case.transB, case.alpha, A, B, case.beta,
                         C if case.beta != 0 else None)


# --------------------------------------------------------------- workloads
SMALL_CASES = [W.SMALL_256, W.SQUARE_1024, W.SWEEP[0], W.SWEEP[1], W.RAGGED[0], W.RAGGED[2]]
LARGE_CASES = [W.SWEEP[2], W.SWEEP[3], W.NT_4096, W.RAGGED[1]]


@pytest.mark.parametrize("algo", ["auto", "simt_cpasync", "tc_3xtf32", "small"])
@pytest.mark.parametrize("case", SMALL_CASES, ids=[c.name for c in SMALL_CASES])
def test_workload_full(orc, case, algo):
    G, (A, B, C) = run_case(case, algo=algo)
    R = oracle_full(orc, case, A, B, C)
    assert_close(G, R, case.K, case.name)


@pytest.mark.parametrize("algo", ["auto", "tc_3xtf32", "small"])
@pytest.mark.parametrize("case", SMALL_CASES, ids=[c.name for c in SMALL_CASES])
def test_workload_integer_bit_exact(orc, case, algo):
    ic = case.as_int()
    G, (A, B, C) = run_case(ic, algo=algo)
    assert_bit_exact(G, oracle_full(orc, ic, A, B, C), ic.name)


class _OracleCache:
    """Seeded inputs and the oracle's whole FP64 result of one full-size case,
    kept for the module so that the two kernel families share one oracle run
    (4096^3 takes about 2 s on 16 host cores)."""

    def __init__(self):
        self.key, self.value = None, None

    def get(self, orc, case):
        if self.key != case.name:
            self.key, self.value = None, None   # free the previous case first
            A, B, C = W.make_inputs(case)
            R = oracle_full(orc, case, A.numpy(), B.numpy(), C.numpy())
            self.key, self.value = case.name, ((A, B, C), R)
        return self.value


_full_cache = _OracleCache()


# (the case varies slowest, so that both families reuse one oracle result)
@pytest.mark.parametrize("algo", ["auto", "tc_3xtf32"])
@pytest.mark.parametrize("case", LARGE_CASES, ids=[c.name for c in LARGE_CASES])
def test_workload_full_size(orc, case, algo):
    """Every one of the M x N outputs of the full-size workloads (2048^3 and
    4096^3 NN, 4096^3 NT with alpha 1.5 and beta 0.5, 8192 x 64 x 4096 with
    beta 1) against the FP64 oracle: relative Frobenius error and the largest
    elementwise error over the whole matrix."""
    (A, B, C), R = _full_cache.get(orc, case)
    G, _ = run_case(case, algo=algo, A=A, B=B, C=C)
    assert_close(G, R, case.K, f"{case.name} {algo}")


@pytest.mark.parametrize("algo", ["auto", "tc_3xtf32"])
@pytest.mark.parametrize("case", [c.as_int() for c in LARGE_CASES],
                         ids=[c.name + "_int" for c in LARGE_CASES])
def test_workload_integer_full_size_bit_exact(orc, case, algo):
    """The same shapes, ops and scalars with random integer A, B and C in
    [-8, 8]: every output equals the oracle bit for bit."""
    (A, B, C), R = _full_cache.get(orc, case)
    G, _ = run_case(case, algo=algo, A=A, B=B, C=C)
    assert_bit_exact(G, R, f"{case.name} {algo}")


@pytest.mark.parametrize("algo", ["auto", "tc_3xtf32"])
def test_full_size_integer_row_sums(algo):
    """A property that holds at any size: with all-ones op(B), every output of
    row i is alpha * sum_k op(A)[i, k] (exact for small integers), checked over
    the whole 4096^3 output."""
    M = N = K = 4096
    g = torch.Generator().manual_seed(7)
    A = torch.randint(-8, 9, (M, K), generator=g).float()
    B = torch.ones((K, N))
    dC = torch.empty((M, N), device="cuda")
    sg.gemm(A.cuda(), B.cuda(), dC, 1.0, 0.0, algo=algo)
    want = A.double().sum(1, keepdim=True).expand(M, N)
    assert torch.equal(dC.cpu().double(), want)


# --------------------------------------------------------------- op/algo grid
SHAPES = [(1, 1, 1), (7, 3, 5), (128, 128, 32), (127, 129, 33), (300, 260, 200),
          (129, 257, 97), (64, 400, 31), (513, 70, 64), (256, 384, 1000)]


@pytest.mark.parametrize("algo", ALL_ALGOS)
@pytest.mark.parametrize("op", OPS, ids=["NN", "NT", "TN", "TT"])
def test_ops_shapes(orc, algo, op):
    ta, tb = op
    for idx, (M, N, K) in enumerate(SHAPES):
        seed = 1000 + idx
        case = W.Case(f"grid_{M}x{N}x{K}", M, N, K, ta, tb, "uniform", seed, 1.25, -0.5)
        G, (A, B, C) = run_case(case, algo=algo)
        assert_close(G, oracle_full(orc, case, A, B, C), K, f"{algo} {op} {M}x{N}x{K}")
        ic = case.as_int()
        G, (A, B, C) = run_case(ic, algo=algo)
        assert_bit_exact(G, oracle_full(orc, ic, A, B, C), f"{algo} {op} int {M}x{N}x{K}")


@pytest.mark.parametrize("algo", GEMM_ALGOS)
def test_random_ragged_sweep(orc, algo):
    """A few dozen random shapes 1..300 per dimension, random ops, scalars and
    padded leading dimensions (the pages' advice: compare many random shapes
    with a CPU reference)."""
    rng = np.random.default_rng({"simt_tma": 42, "simt_cpasync": 43, "small": 45, "reg_2x2": 46,
                                 "reg_4x4": 47}.get(algo, 44))
    for t in range(40):
        M, N, K = (int(x) for x in rng.integers(1, 301, size=3))
        ta, tb = int(rng.integers(0, 2)), int(rng.integers(0, 2))
        alpha = float(rng.choice([1.0, -0.5, 2.0, 0.75]))
        beta = float(rng.choice([0.0, 1.0, -1.5]))
        case = W.Case("sweep", M, N, K, ta, tb, "uniform", 5000 + t, alpha, beta)
        A, B, C = W.make_inputs(case)
        if algo in ANY_LAYOUT_ALGOS:   # any padding, ld usually not a multiple of 4
            ea, eb = int(rng.integers(0, 5)), int(rng.integers(0, 5))
        else:                        # pad each ld up to a multiple of 4 (TMA needs 16-byte rows)
            ea = (-A.shape[1]) % 4 + 4 * int(rng.integers(0, 3))
            eb = (-B.shape[1]) % 4 + 4 * int(rng.integers(0, 3))
        Ad, Bd = padded(A.cuda(), ea), padded(B.cuda(), eb)
        Cd = padded(C.cuda(), int(rng.integers(0, 3)), fill=float("nan") if beta == 0 else 0.0)
        sg.gemm(Ad, Bd, Cd, alpha, beta, ta, tb, algo=algo)
        torch.cuda.synchronize()
        R = orc.sgemm_f64(ta, tb, alpha, A.numpy(), B.numpy(), beta, C.numpy() if beta else None)
        assert_close(Cd.cpu().numpy(), R, K, f"{algo} t={t} {M}x{N}x{K} op={ta}{tb}")


# --------------------------------------------------------------- layout edge cases
def test_guard_bands_untouched(orc):
    """Nothing outside the M x N output (inside ldc) is written."""
    M, N, K = 200, 130, 72
    for algo in ALL_ALGOS:
        A = torch.rand(M, K, device="cuda")
        B = padded(torch.rand(K, N, device="cuda"), 2)   # ldb = 132: TMA-eligible
        big = torch.full((M + 3, N + 5), 12345.0, device="cuda")
        C = big[:M, :N]
        sg.gemm(A, B, C, 1.0, 0.0, algo=algo)
        torch.cuda.synchronize()
        assert torch.all(big[:M, N:] == 12345.0), algo
        assert torch.all(big[M:, :] == 12345.0), algo
        R = orc.sgemm_f64(0, 0, 1.0, A.cpu().numpy(), B.cpu().numpy())
        assert_close(C.cpu().numpy(), R, K, algo)


# (M, N, K, transA, transB): 128 x 128 tiles with beta = 0, ragged in M;
# N % 4 == 0 takes the staged TMA stores, the odd N the register epilogue
# (a TMA store would write the rest of the last 16-byte granule of a row)
STAGED = [(1000, 700, 300, 0, 0), (1003, 1004, 512, 1, 0), (777, 1996, 96, 1, 1),
          (1003, 1001, 512, 1, 0), (777, 1999, 96, 1, 1)]


@pytest.mark.parametrize("case", STAGED, ids=["NN", "TN", "TT", "TN_odd_N", "TT_odd_N"])
def test_staged_epilogue_guard_bands(orc, case):
    """Tiles staged in shared memory and written by TMA stores: every output
    equals the oracle's within tolerance and nothing outside M x N (inside
    ldc, or past the last row) is written -- the stores clip the ragged
    tiles."""
    M, N, K, ta, tb = case
    g = torch.Generator().manual_seed(M + N)
    A = torch.rand((K, M) if ta else (M, K), generator=g).mul_(2).sub_(1)
    B = torch.rand((N, K) if tb else (K, N), generator=g).mul_(2).sub_(1)
    dA, dB = padded(A.cuda(), (-A.shape[1]) % 4, 0.0), padded(B.cuda(), (-B.shape[1]) % 4, 0.0)
    ldc = N + (-N) % 4 + 4
    big = torch.full((M + 2, ldc), 12345.0, device="cuda")
    C = big[:M, :N]
    sg.gemm(dA, dB, C, 1.5, 0.0, ta, tb)
    torch.cuda.synchronize()
    assert torch.all(big[:M, N:] == 12345.0)
    assert torch.all(big[M:, :] == 12345.0)
    assert_close(C.cpu().numpy(), orc.sgemm_f64(ta, tb, 1.5, A.numpy(), B.numpy()), K, f"staged {case}")


@pytest.mark.parametrize("op", OPS, ids=["NN", "NT", "TN", "TT"])
def test_misaligned_pointers_use_cpasync(orc, op):
    ta, tb = op
    M, N, K = 650, 420, 270      # above the small-product kernel's range
    case = W.Case("mis", M, N, K, ta, tb, "uniform", 77, 1.0, 1.0)
    A, B, C = W.make_inputs(case)
    Ad, Bd = offset_view(A.cuda(), 1), offset_view(B.cuda(), 3)
    Cd = offset_view(C.cuda(), 2)
    assert sg.sgemm_select_algo(ta, tb, M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(),
                                Bd.stride(0), 1.0, 1.0, Cd.data_ptr(), N) == sg.ALGO_SIMT_CPASYNC
    for algo in TMA_ALGOS:
        with pytest.raises(sg.SgemmError):
            sg.gemm(Ad, Bd, Cd, 1.0, 1.0, ta, tb, algo=algo)
    sg.gemm(Ad, Bd, Cd, 1.0, 1.0, ta, tb)
    torch.cuda.synchronize()
    R = orc.sgemm_f64(ta, tb, 1.0, A.numpy(), B.numpy(), 1.0, C.numpy())
    assert_close(Cd.cpu().numpy(), R, K, f"misaligned {op}")
    # the comparison kernels fall back to element loads and stores
    for algo in ("reg_2x2", "reg_4x4"):
        Cd = offset_view(C.cuda(), 2)
        sg.gemm(Ad, Bd, Cd, 1.0, 1.0, ta, tb, algo=algo)
        torch.cuda.synchronize()
        assert_close(Cd.cpu().numpy(), R, K, f"misaligned {op} {algo}")


def test_odd_leading_dimensions_are_repacked(orc):
    """The pages' ragged configuration: lda = K = 997, ldb = N = 1013 (TMA-ineligible).
    Forcing the TMA family is refused; AUTO copies both operands into aligned
    scratch (two repack launches) and runs the TMA kernel, which it reports."""
    case = W.RAGGED[0]
    A, B, C = (t.cuda() for t in W.make_inputs(case))
    assert sg.sgemm_select_algo(0, 0, case.M, case.N, case.K, A.data_ptr(), case.K, B.data_ptr(),
                                case.N, 1.0, 1.0, C.data_ptr(), case.N) == sg.ALGO_SIMT_TMA
    with pytest.raises(sg.SgemmError):
        sg.gemm(A, B, C, 1.0, 1.0, algo="simt_tma")
    C0 = C.clone()
    sg.gemm(A, B, C, case.alpha, case.beta)
    n = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    Ap, Bp = padded(A, (-case.K) % 4), padded(B, (-case.N) % 4)
    C2 = C0.clone()
    sg.gemm(Ap, Bp, C2, case.alpha, case.beta, algo="simt_tma")
    torch.cuda.synchronize()
    assert torch.equal(C, C2)
    assert n == sg.sgemm_last_launch_count() + 1   # one launch repacks both


# (M, N, K, transA, transB, A offset, B offset): odd leading dimensions and
# misaligned bases, each operand repacked or (where the plan transposes it
# anyway) transposed from its unaligned storage
REPACK_CASES = [(1000, 1013, 997, 1, 1, 0, 0), (700, 1500, 999, 0, 1, 1, 0),
                (2048, 2048, 1023, 0, 0, 0, 0), (2048, 2052, 1021, 0, 1, 3, 2),
                (1500, 333, 2000, 1, 0, 2, 1)]


@pytest.mark.parametrize("case", REPACK_CASES, ids=lambda c: "x".join(map(str, c)))
def test_repacked_operands_match_aligned_call(orc, case):
    """An AUTO product on TMA-ineligible operands equals, bit for bit, the same
    call on aligned copies of them (same kernel, same tiles, same k order);
    sampled outputs also meet the FP32 tolerance against the oracle."""
    M, N, K, ta, tb, oa, ob = case
    g = torch.Generator().manual_seed(M + 3 * N + K)
    A = torch.rand((K, M) if ta else (M, K), generator=g).mul_(2).sub_(1)
    B = torch.rand((N, K) if tb else (K, N), generator=g).mul_(2).sub_(1)
    C0 = torch.rand(M, N, generator=g).cuda()
    dA = offset_view(A.cuda(), oa) if oa else A.cuda()
    dB = offset_view(B.cuda(), ob) if ob else B.cuda()
    assert sg.sgemm_select_algo(ta, tb, M, N, K, dA.data_ptr(), dA.stride(0), dB.data_ptr(),
                                dB.stride(0), 0.5, 1.5, C0.data_ptr(), N) == sg.ALGO_SIMT_TMA
    C1 = C0.clone()
    sg.gemm(dA, dB, C1, 0.5, 1.5, ta, tb)
    n1 = sg.sgemm_last_launch_count()
    Ap = padded(A.cuda(), (-A.shape[1]) % 4)
    Bp = padded(B.cuda(), (-B.shape[1]) % 4)
    C2 = C0.clone()
    sg.gemm(Ap, Bp, C2, 0.5, 1.5, ta, tb, algo="simt_tma")
    n2 = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    # at most one repack launch (both operands) and a transpose of a
    # misaligned operand the aligned call transposes too
    assert n2 <= n1 <= n2 + 1
    I, J = sample_indices(M, N, 2000, seed=K)
    R = orc.sgemm_entries_f64(ta, tb, 0.5, A.numpy(), B.numpy(), 1.5, C0.cpu().numpy(), I, J)
    assert_close(C1.cpu().numpy()[I, J], R, K, f"repacked {case}")


# --------------------------------------------------------------- degenerate cases
@pytest.mark.parametrize("algo", ALL_ALGOS)
def test_beta_zero_ignores_nan_in_c(orc, algo):
    M, N, K = 70, 92, 52
    A = torch.rand(M, K, device="cuda")
    B = torch.rand(K, N, device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    sg.gemm(A, B, C, 1.0, 0.0, algo=algo)
    torch.cuda.synchronize()
    R = orc.sgemm_f64(0, 0, 1.0, A.cpu().numpy(), B.cpu().numpy())
    assert_close(C.cpu().numpy(), R, K, algo)


def test_alpha_zero_and_k_zero():
    M, N = 33, 47
    C0 = torch.rand(M, N, device="cuda")
    A = torch.full((M, 8), float("nan"), device="cuda")
    B = torch.full((8, N), float("nan"), device="cuda")
    C = C0.clone()
    sg.gemm(A, B, C, 0.0, 2.0)
    torch.cuda.synchronize()
    assert torch.equal(C, 2.0 * C0)
    C = C0.clone()
    sg.gemm(A, B, C, 0.0, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))
    C = torch.full((M, N), float("nan"), device="cuda")
    Ak = torch.empty((M, 0), device="cuda")
    Bk = torch.empty((0, N), device="cuda")
    sg.gemm(Ak, Bk, C, 1.0, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))
    assert sg.sgemm_last_launch_count() == 1


def test_empty_outputs():
    A = torch.rand(0, 5, device="cuda")
    B = torch.rand(5, 7, device="cuda")
    C = torch.empty(0, 7, device="cuda")
    sg.gemm(A, B, C)
    assert sg.sgemm_last_launch_count() == 0


# (M, N, K): one CTA per tile for the tensor-core family at the first two;
# at the third it splits the operands ahead and runs on CTA pairs
SUBNORMAL_SHAPES = [(128, 128, 128), (256, 384, 160), (2048, 2560, 512)]
SUBNORMAL_ALGOS = ["auto", "simt_tma", "simt_cpasync", "tc_3xtf32", "naive", "smem_tiled",
                   "small", "reg_2x2", "reg_4x4"]


def _small_ints(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-8, 9, shape, generator=g).float()


@pytest.mark.parametrize("shape", SUBNORMAL_SHAPES, ids=["%dx%dx%d" % s for s in SUBNORMAL_SHAPES])
def test_subnormals_are_kept(orc, shape):
    """No family flushes subnormals, the 3xTF32 tensor-core path included:
    (1) normal inputs whose products and sums are subnormal (integers times
    2^-70 on both sides: results are integers times 2^-140) and (2) subnormal
    inputs whose significant bits fit TF32's 10-bit mantissa (integers times
    2^-135) against normal ones (integers times 2^100) give every output
    bit for bit equal to the oracle."""
    M, N, K = shape
    ai, bi = _small_ints((M, K), M + K), _small_ints((K, N), N + 1)
    for A, B, what in ((ai * 2.0 ** -70, bi * 2.0 ** -70, "subnormal results"),
                       (ai * 2.0 ** -135, bi * 2.0 ** 100, "subnormal inputs")):
        R = orc.sgemm_f64(0, 0, 1.0, A.numpy(), B.numpy())
        assert np.any((R != 0) & (np.abs(R) < 2.0 ** -126)) or what == "subnormal inputs"
        dA, dB = A.cuda(), B.cuda()
        for algo in SUBNORMAL_ALGOS:
            if algo in ("naive", "smem_tiled") and M * N * K > 1 << 24:
                continue
            C = torch.empty(M, N, device="cuda")
            sg.gemm(dA, dB, C, 1.0, 0.0, algo=algo)
            torch.cuda.synchronize()
            assert_bit_exact(C.cpu().numpy(), R, f"{what} {algo} {shape}")


@pytest.mark.parametrize("shape", [SUBNORMAL_SHAPES[0], SUBNORMAL_SHAPES[2]], ids=["one_cta", "pairs"])
def test_subnormal_inputs_beyond_tf32_resolution(orc, shape):
    """Subnormal inputs with all 23 mantissa bits (random bit patterns) against
    integers times 2^100.  The CUDA-core families meet the FP32 tolerance on
    the (normal-range) results.  The 3xTF32 path represents each such input
    as big + small TF32 parts, whose subnormal spacing is 2^-136: every input
    is kept to within 2^-137, so |G - R| <= 2^-137 * sum_k |b_kj| (plus FP32
    rounding of the sums) for every output -- up to about 2^-10 relative, a
    documented precision loss of that family on subnormal inputs."""
    M, N, K = shape
    g = torch.Generator().manual_seed(11)
    bits = torch.randint(1, 1 << 23, (M, K), generator=g, dtype=torch.int32)
    bits |= torch.randint(0, 2, (M, K), generator=g, dtype=torch.int32) << 31
    A = bits.view(torch.float32)
    assert torch.all(A.abs() < 2.0 ** -126) and torch.all(A != 0)
    B = _small_ints((K, N), 12) * 2.0 ** 100
    R = orc.sgemm_f64(0, 0, 1.0, A.numpy(), B.numpy())
    absB = np.abs(B.numpy().astype(np.float64))
    absAB = np.abs(A.numpy().astype(np.float64)) @ absB
    bound = 2.0 ** -137 * absB.sum(axis=0)[None, :] + 2.0 ** -20 * absAB
    dA, dB = A.cuda(), B.cuda()
    for algo in ["auto", "simt_tma", "simt_cpasync", "small", "reg_4x4", "tc_3xtf32"]:
        C = torch.empty(M, N, device="cuda")
        sg.gemm(dA, dB, C, 1.0, 0.0, algo=algo)
        torch.cuda.synchronize()
        G = C.cpu().numpy().astype(np.float64)
        if algo == "tc_3xtf32":
            worst = float(np.max(np.abs(G - R) - bound))
            assert worst <= 0, f"{algo} {shape}: exceeds the bound by {worst:.3e}"
        else:
            rel = np.linalg.norm(G - R) / np.linalg.norm(R)
            assert rel <= 1e-5, f"{algo} {shape}: rel_fro {rel:.3e}"


# --------------------------------------------------------------- streams / status
def test_runs_on_the_given_stream(orc):
    s = torch.cuda.Stream()
    M, N, K = 512, 512, 512
    A = torch.rand(M, K, device="cuda")
    B = torch.rand(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    with torch.cuda.stream(s):
        sg.gemm(A, B, C)
    s.synchronize()
    R = orc.sgemm_f64(0, 0, 1.0, A.cpu().numpy(), B.cpu().numpy())
    assert_close(C.cpu().numpy(), R, K, "side stream")


@pytest.mark.parametrize("shape", [(512, 512, 512), (1024, 1024, 1024), (2048, 2048, 256),
                                   (8192, 64, 1024)], ids=lambda s: "x".join(map(str, s)))
def test_products_see_the_previous_kernels_writes(shape):
    """Product kernels are launched as programmatic dependents of whatever
    kernel precedes them on the stream, and touch memory only once that kernel
    has finished.  Each call here directly follows kernels (torch's) that
    rewrite A and B and scale C, and the next rewrite directly follows the
    product: every result equals the same product run in isolation, bit for
    bit (integer-valued data: exact in any order)."""
    M, N, K = shape
    g = torch.Generator().manual_seed(M + N + K)
    As = [torch.randint(-4, 5, (M, K), generator=g).float().cuda() for _ in range(3)]
    Bs = [torch.randint(-4, 5, (K, N), generator=g).float().cuda() for _ in range(3)]
    ref = []
    for a, b in zip(As, Bs):
        c = torch.full((M, N), 3.0, device="cuda")
        sg.gemm(a, b, c, 1.0, 0.5)
        torch.cuda.synchronize()
        ref.append(c.clone())
    A = torch.empty(M, K, device="cuda")
    B = torch.empty(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    outs = []
    for it in range(6):
        i = it % 3
        A.copy_(As[i])
        B.copy_(Bs[i])
        C.fill_(3.0)
        sg.gemm(A, B, C, 1.0, 0.5)
        outs.append(C.clone())
    torch.cuda.synchronize()
    for it, c in enumerate(outs):
        assert torch.equal(c, ref[it % 3]), f"call {it}"


def test_launch_count_single_k_slice_is_one():
    """K = 32 is one k-slice: nothing to split, one launch for every family."""
    A = torch.rand(300, 32, device="cuda")
    B = torch.rand(32, 100, device="cuda")
    for algo in ALL_ALGOS:
        sg.gemm(A, B, algo=algo)
        assert sg.sgemm_last_launch_count() == 1, algo


def test_bounded_wait_gives_up_and_context_survives(orc):
    """A wait that nothing satisfies ends with SGEMM_ERR_DEVICE_TIMEOUT in about
    the given budget; the next GEMM on the same context is still correct."""
    import time
    assert sg.sgemm_last_device_status() == 0
    t0 = time.perf_counter()
    sg.sgemm_selftest_wait_timeout(2_000_000)       # 2 ms
    st = sg.sgemm_last_device_status()
    assert st == 5, st
    assert time.perf_counter() - t0 < 5.0
    assert sg.sgemm_last_device_status() == 0       # cleared by the read
    A = torch.rand(256, 256, device="cuda")
    B = torch.rand(256, 256, device="cuda")
    C = sg.gemm(A, B)
    torch.cuda.synchronize()
    assert_close(C.cpu().numpy(), orc.sgemm_f64(0, 0, 1.0, A.cpu().numpy(), B.cpu().numpy()), 256,
                 "after timeout")


# --------------------------------------------------------------- stream-K split
SK_SHAPES = [(1024, 1024, 1024), (2048, 2048, 2048), (8192, 64, 4096), (256, 384, 1000),
             (4096, 4096, 4096)]


@pytest.mark.parametrize("shape", SK_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SK_SHAPES])
def test_stream_k_is_deterministic(shape):
    """Tiles whose k-iterations are spread over several CTAs are summed in a
    fixed order: repeated runs give bit-identical results."""
    M, N, K = shape
    g = torch.Generator().manual_seed(99)
    A = torch.randn(M, K, generator=g).cuda()
    B = torch.randn(K, N, generator=g).cuda()
    C0 = torch.randn(M, N, generator=g).cuda()
    outs = []
    for _ in range(3):
        C = C0.clone()
        sg.gemm(A, B, C, 0.5, 2.0)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_stream_k_launches():
    """Large products finish split tiles inside the product kernel (the CTA
    that arrives last at a tile adds its partials): one launch.  Tiles split
    into many segments take the separate fixup pass: two launches.  Products
    whose tiles fit in clusters of two or more CTAs split each tile inside its
    cluster: one launch."""
    A = torch.randn(2048, 2048, device="cuda")
    B = torch.randn(2048, 2048, device="cuda")
    sg.gemm(A, B, transA=True)                  # TN: no operand transposed ahead
    assert sg.sgemm_last_launch_count() == 1
    A = torch.randn(1280, 1024, device="cuda")
    B = torch.randn(1024, 1024, device="cuda")
    sg.gemm(A, B)                               # 80 tiles over every SM, A transposed in smem
    assert sg.sgemm_last_launch_count() == 2
    A = torch.randn(512, 512, device="cuda")
    B = torch.randn(512, 1024, device="cuda")
    sg.gemm(A, B, transA=True)                  # 32 tiles of 16 k-tiles: clusters
    assert sg.sgemm_last_launch_count() == 1
    A = torch.randn(128 * 152, 256, device="cuda")
    B = torch.randn(256, 128, device="cuda")
    sg.gemm(A, B)                               # exactly one wave of whole tiles
    assert sg.sgemm_last_launch_count() == 1


# (M, N, K, transA, transB): products with fewer tiles than CTA slots and
# short k-ranges, split over the CTAs of a cluster (each tile's k-tiles in S
# shares, S = 2 or 4) and reduced through distributed shared memory; 128 x 64
# and 128 x 128 tiles, ragged in M, N and K, K not a multiple of S k-tiles
CSK_SHAPES = [(512, 512, 512, 0, 0), (700, 650, 500, 0, 1), (300, 260, 1000, 1, 0),
              (1024, 1024, 512, 1, 1), (129, 1000, 1000, 0, 0), (640, 640, 640, 0, 0)]


@pytest.mark.parametrize("shape", CSK_SHAPES, ids=["%dx%dx%d_%s%s" % (s[0], s[1], s[2], "NT"[s[3]], "NT"[s[4]])
                                                 for s in CSK_SHAPES])
def test_cluster_split_k(orc, shape):
    """One launch; every output against the oracle (random inputs, alpha and
    beta) and bit for bit on integer inputs; the same bits on a second run;
    through the TMA and the cp.async producers."""
    M, N, K, ta, tb = shape
    case = W.Case("csk", M, N, K, ta, tb, "uniform", 700 + M, 1.25, -0.75)
    for algo in ("auto", "simt_cpasync"):
        G, (A, B, C) = run_case(case, algo=algo)
        assert sg.sgemm_last_launch_count() == 1, algo
        R = oracle_full(orc, case, A, B, C)
        assert_close(G, R, K, f"cluster split-K {shape} {algo}")
        G2, _ = run_case(case, algo=algo, A=torch.from_numpy(A), B=torch.from_numpy(B), C=torch.from_numpy(C))
        assert np.array_equal(G, G2), f"{shape} {algo}: not deterministic"
        ic = case.as_int()
        Gi, (Ai, Bi, Ci) = run_case(ic, algo=algo)
        assert_bit_exact(Gi, oracle_full(orc, ic, Ai, Bi, Ci), f"cluster split-K int {shape} {algo}")


# --------------------------------------------------------------- operands transposed ahead
PRE_SHAPES = [(2048, 4864, 256), (2502, 4100, 300), (2048, 2048, 2048)]


@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 1)], ids=["NN", "NT", "TT"])
@pytest.mark.parametrize("shape", PRE_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in PRE_SHAPES])
def test_pretransposed_matches_tn_bit_for_bit(shape, op):
    """Large NN / NT / TT products (TMA-eligible, at least one 128 x 256 tile
    per SM) have their k-contiguous operand(s) transposed into scratch first
    and then run as TN: the result must equal, bit for bit, the TN call on
    operands transposed by torch (same kernel, same tiles, same k order), with
    one extra launch per transposed operand.  An operand whose rows are not
    16-byte aligned is copied into aligned scratch even when not transposed
    (one launch too)."""
    M, N, K = shape
    ta, tb = op
    g = torch.Generator().manual_seed(M + N + K + 2 * ta + tb)
    A = torch.randn((K, M) if ta else (M, K), generator=g).cuda()
    B = torch.randn((N, K) if tb else (K, N), generator=g).cuda()
    C0 = torch.randn(M, N, generator=g).cuda()
    C1 = C0.clone()
    sg.gemm(A, B, C1, 0.75, 0.5, ta, tb)
    n1 = sg.sgemm_last_launch_count()
    # K x M and K x N, rows padded to 16 bytes as the library's scratch is, so
    # that the reference call takes the same (TMA) kernel
    At = padded(A if ta else A.t().contiguous(), (-M) % 4)
    Bn = padded(B.t().contiguous() if tb else B, (-N) % 4)
    C2 = C0.clone()
    sg.gemm(At, Bn, C2, 0.75, 0.5, 1, 0)
    n2 = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    # transposed ahead at GPU-filling size; a misaligned operand is copied anyway
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = M * N * K >= 2 ** 30 and -(-M // 128) * -(-N // 256) * 100 >= 40 * sms
    t_a, t_b = big and ta == 0 and N >= 1024, big and tb == 1 and M >= 1024
    a_ok, b_ok = A.stride(0) % 4 == 0, B.stride(0) % 4 == 0
    # one launch per transposed operand, one for any operands only repacked
    copies = t_a + t_b + ((not a_ok and not t_a) or (not b_ok and not t_b))
    assert n1 == n2 + copies


@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 1)], ids=["NN", "NT", "TT"])
def test_tensor_core_pretransposed_matches_tn_bit_for_bit(op):
    """Large 3xTF32 products split both operands ahead (a pass per operand,
    transposing an m/n-contiguous one to K-major) and run the converter-free
    kernel: NN / NT / TT must equal, bit for bit, the TN call on operands
    transposed by torch, and take three launches."""
    M, N, K = 2048, 2560, 512
    ta, tb = op
    g = torch.Generator().manual_seed(11 + 2 * ta + tb)
    A = torch.randn((K, M) if ta else (M, K), generator=g).cuda()
    B = torch.randn((N, K) if tb else (K, N), generator=g).cuda()
    C1 = torch.empty(M, N, device="cuda")
    sg.gemm(A, B, C1, 1.0, 0.0, ta, tb, algo="tc_3xtf32")
    n1 = sg.sgemm_last_launch_count()
    At = A if ta else A.t().contiguous()
    Bn = B.t().contiguous() if tb else B
    C2 = torch.empty(M, N, device="cuda")
    sg.gemm(At, Bn, C2, 1.0, 0.0, 1, 0, algo="tc_3xtf32")
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    assert n1 == 3 and sg.sgemm_last_launch_count() == 3


@pytest.mark.parametrize("op", [(0, 0), (1, 1)], ids=["NN", "TT"])
def test_tensor_core_split_ahead_ragged(orc, op):
    """Split ahead on a product whose M and N end in partial tiles, with alpha
    and beta (C read): sampled outputs against the oracle; and a TMA-eligible
    product with K % 4 != 0 (rows padded), which keeps the in-kernel split."""
    ta, tb = op
    for (M, N, K, pad) in [(2000, 2504, 1004, 0), (2048, 2560, 1002, 2)]:
        g = torch.Generator().manual_seed(M + K + ta)
        A = torch.rand((K, M) if ta else (M, K), generator=g).mul_(2).sub_(1)
        B = torch.rand((N, K) if tb else (K, N), generator=g).mul_(2).sub_(1)
        C0 = torch.rand(M, N, generator=g).mul_(2).sub_(1)
        dA = padded(A.cuda(), pad) if not ta else A.cuda()
        dB = padded(B.cuda(), pad) if tb else B.cuda()
        dC = C0.cuda()
        sg.gemm(dA, dB, dC, 1.25, -0.5, ta, tb, algo="tc_3xtf32")
        n = sg.sgemm_last_launch_count()
        torch.cuda.synchronize()
        assert n == (3 if K % 4 == 0 else n)
        I, J = sample_indices(M, N, 3000, seed=M)
        R = orc.sgemm_entries_f64(ta, tb, 1.25, A.numpy(), B.numpy(), -0.5, C0.numpy(), I, J)
        G = dC.cpu().numpy()[I, J]
        assert_close(G, R, K, f"tc split ahead {M}x{N}x{K} {op}")


@pytest.mark.parametrize("N", [2500, 2400])
def test_tensor_core_wide_tiles_ragged(orc, N):
    """Split-ahead 3xTF32 products of this shape run whole 256-wide tiles
    whose two 128-column halves are written by separate epilogue
    warpgroups.  N = 2500 ends in a partly filled second half, N =
    2400 in a second half wholly past N (its op(B) box reads only fill
    values).  Rows depend only on their own tile row: the rows that an M =
    1792 and an M = 1664 product of the same operands share agree bit for
    bit.  Sampled outputs are checked against the oracle, with alpha and beta
    (C read)."""
    K = 512
    g = torch.Generator().manual_seed(N)
    A = torch.randn(1792, K, generator=g)
    B = torch.randn(K, N, generator=g)
    C0 = torch.rand(1792, N, generator=g).mul_(2).sub_(1)
    dA, dB = A.cuda(), B.cuda()
    C_full, C_part = C0.cuda(), C0[:1664].cuda()
    sg.gemm(dA, dB, C_full, 0.75, 0.5, 0, 0, algo="tc_3xtf32")
    n_full = sg.sgemm_last_launch_count()
    sg.gemm(dA[:1664], dB, C_part, 0.75, 0.5, 0, 0, algo="tc_3xtf32")
    n_part = sg.sgemm_last_launch_count()
    torch.cuda.synchronize()
    assert n_full == 3 and n_part == 3
    assert torch.equal(C_full[:1664], C_part)
    I, J = sample_indices(1792, N, 3000, seed=N)
    J[:200] = np.arange(N - 200, N)   # the ragged last tile's columns
    R = orc.sgemm_entries_f64(0, 0, 0.75, A.numpy(), B.numpy(), 0.5, C0.numpy(), I, J)
    assert_close(C_full.cpu().numpy()[I, J], R, K, f"tc wide tiles N={N}")


PAIR_CASES = [(1792, 1664, 4000), (1792, 1600, 4000), (2048, 1920, 2432)]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tensor_core_cta_pairs(orc, case):
    """Split-ahead products run on CTA pairs (tcgen05 cta_group::2): 256-row
    tiles, each CTA holding its 128 rows of A and half of op(B)'s columns.
    N = 4000 takes whole 256 x 256 tiles for a full round of pairs and column
    halves for the rest; N = 2432 (19 column tiles of 128) takes 256 x 128
    tiles.  M = 1664 (13 row tiles) leaves the last pair's second CTA wholly
    below the matrix (its A boxes read only fill values), M = 1600 and 1920
    partly.  Rows agree bit for bit with the same rows of a product with more
    rows (every pair full) of the same operands, and sampled outputs match the
    oracle, with alpha and beta (C read) and a ragged N."""
    M_full, M, N = case
    K = 512
    g = torch.Generator().manual_seed(M + N)
    A = torch.randn(M_full, K, generator=g)
    B = torch.randn(K, N, generator=g)
    C0 = torch.rand(M_full, N, generator=g).mul_(2).sub_(1)
    dA, dB = A.cuda(), B.cuda()
    C_full, C_part = C0.cuda(), C0[:M].cuda()
    sg.gemm(dA, dB, C_full, 1.5, -0.5, 0, 0, algo="tc_3xtf32")
    sg.gemm(dA[:M], dB, C_part, 1.5, -0.5, 0, 0, algo="tc_3xtf32")
    assert sg.sgemm_last_launch_count() == 3
    torch.cuda.synchronize()
    assert torch.equal(C_full[:M], C_part)
    I, J = sample_indices(M, N, 3000, seed=M)
    R = orc.sgemm_entries_f64(0, 0, 1.5, A[:M].numpy(), B.numpy(), -0.5, C0[:M].numpy(), I, J)
    assert_close(C_part.cpu().numpy()[I, J], R, K, f"tc CTA pairs {case}")


def test_pretransposed_on_two_streams(orc):
    """Calls on different streams share the transposed-operand scratch; the
    library orders them, so every result is right."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.Generator().manual_seed(6)
    mats = [(torch.randn(2048, 512, generator=g), torch.randn(512, 4864, generator=g))
            for _ in range(2)]
    dev = [(a.cuda(), b.cuda(), torch.empty(2048, 4864, device="cuda")) for a, b in mats]
    torch.cuda.synchronize()
    for _ in range(4):
        for (A, B, C), s in zip(dev, (s1, s2)):
            with torch.cuda.stream(s):
                sg.gemm(A, B, C, stream=s)
            assert sg.sgemm_last_launch_count() >= 2
    torch.cuda.synchronize()
    for (a, b), (_, _, C) in zip(mats, dev):
        assert_close(C.cpu().numpy(), orc.sgemm_f64(0, 0, 1.0, a.numpy(), b.numpy()), 512, "stream")


def test_stream_k_on_two_streams(orc):
    """Stream-K calls on different streams share the device workspace; the
    library orders them, so both results are right."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.Generator().manual_seed(5)
    # 80 tiles of 128 x 128: stream-K with the workspace (too many for clusters)
    mats = [(torch.randn(1280, 1024, generator=g), torch.randn(1024, 1024, generator=g))
            for _ in range(2)]
    dev = [(a.cuda(), b.cuda(), torch.empty(1280, 1024, device="cuda")) for a, b in mats]
    torch.cuda.synchronize()
    for _ in range(5):
        with torch.cuda.stream(s1):
            sg.gemm(*dev[0])
        with torch.cuda.stream(s2):
            sg.gemm(*dev[1])
    torch.cuda.synchronize()
    for (a, b), (_, _, c) in zip(mats, dev):
        assert_close(c.cpu().numpy(), orc.sgemm_f64(0, 0, 1.0, a.numpy(), b.numpy()), 1024, "two streams")
