"""The C-ABI library without a GPU: it loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before any CUDA
call (nothing here launches a kernel)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_10_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^SGEMM_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("sgemm", "sgemm_ex", "sgemm_last_device_status", "sgemm_status_string"):
        assert required in names


@pytest.mark.parametrize("name", declared_functions())
def test_symbol_exported(lib, name):
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_only_abi_symbols_exported(lib):
    """-fvisibility=hidden: the dynamic symbol table holds the ABI, not internals."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    syms = {ln.split()[-1] for ln in out.stdout.splitlines() if ln.strip()}
    ours = {s for s in syms if s.startswith("sgemm")}
    assert ours == set(declared_functions())


def test_strings(lib):
    import dense_fp32_matrix_10_gb300 as g
    assert g.sgemm_status_string(0) == "success"
    assert "overlap" in g.sgemm_status_string(2)
    assert g.sgemm_status_string(99) == "unknown status"
    assert [g.sgemm_algo_name(i) for i in range(9)] == \
        ["auto", "simt_tma", "simt_cpasync", "tc_3xtf32", "naive", "smem_tiled", "small",
         "reg_2x2", "reg_4x4"]
    assert g.sgemm_algo_name(42) == "unknown"
    assert re.match(r"^\d+\.\d+\.\d+$", g.sgemm_version())


# (transA, transB, M, N, K, lda, ldb, ldc, A, B, C, alpha) -> expected status
FAKE_A, FAKE_B, FAKE_C = 0x10000, 0x900000, 0x2000000   # disjoint fake device addresses
BAD = [
    ("bad transA", (2, 0, 4, 4, 4, 4, 4, 4)),
    ("bad transB char", (0, ord("x"), 4, 4, 4, 4, 4, 4)),
    ("negative M", (0, 0, -1, 4, 4, 4, 4, 4)),
    ("negative K", (0, 0, 4, 4, -3, 4, 4, 4)),
    ("M too large", (0, 0, 1 << 31, 4, 4, 4, 4, 4)),
    ("lda < K (N)", (0, 0, 4, 4, 8, 7, 4, 4)),
    ("lda < M (T)", (1, 0, 9, 4, 4, 8, 4, 4)),
    ("ldb < N (N)", (0, 0, 4, 9, 4, 4, 8, 9)),
    ("ldb < K (T)", (0, 1, 4, 4, 6, 6, 5, 4)),
    ("ldc < N", (0, 0, 4, 5, 4, 4, 5, 4)),
]


@pytest.mark.parametrize("name,args", BAD, ids=[b[0] for b in BAD])
def test_invalid_arguments(lib, name, args):
    ta, tb, M, N, K, lda, ldb, ldc = args
    st = lib.sgemm(ta, tb, ctypes.c_int64(M), ctypes.c_int64(N), ctypes.c_int64(K),
                   ctypes.c_float(1.0), ctypes.c_void_p(FAKE_A), ctypes.c_int64(lda),
                   ctypes.c_void_p(FAKE_B), ctypes.c_int64(ldb), ctypes.c_float(0.0),
                   ctypes.c_void_p(FAKE_C), ctypes.c_int64(ldc), None)
    assert st == 1


def _call(lib, ta, tb, M, N, K, A, lda, B, ldb, C, ldc, alpha=1.0, beta=0.0, algo=0):
    return lib.sgemm_ex(ta, tb, ctypes.c_int64(M), ctypes.c_int64(N), ctypes.c_int64(K),
                        ctypes.c_float(alpha), ctypes.c_void_p(A), ctypes.c_int64(lda),
                        ctypes.c_void_p(B), ctypes.c_int64(ldb), ctypes.c_float(beta),
                        ctypes.c_void_p(C), ctypes.c_int64(ldc), None, algo)


def test_null_pointers(lib):
    assert _call(lib, 0, 0, 4, 4, 4, 0, 4, FAKE_B, 4, FAKE_C, 4) == 1
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, 0, 4, FAKE_C, 4) == 1
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, 0, 4) == 1


def test_aliasing(lib):
    # C's byte range [FAKE_A + 16, ...) overlaps A's [FAKE_A, FAKE_A + 64)
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 16, 4) == 2
    # C overlapping B, with B transposed and padded
    assert _call(lib, 0, 1, 4, 4, 4, FAKE_A, 4, FAKE_B, 100, FAKE_B + 4 * 250, 4) == 2
    # touching but not overlapping is fine up to the device check
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 64, 4) in (0, 3)


def test_huge_ranges_do_not_wrap(lib):
    """Byte ranges are computed in 128-bit arithmetic: M = 2^24 rows with
    lda = 2^40 span 2^66 bytes, past int64 and the address space -- refused as
    an impossible matrix instead of wrapping into a small range."""
    big_ld = 1 << 40
    assert _call(lib, 0, 0, 1 << 24, 4, 4, FAKE_A, big_ld, FAKE_B, 4, FAKE_C, 4) == 1
    assert _call(lib, 0, 0, 4, 4, 1 << 24, FAKE_A, 1 << 24, FAKE_B, big_ld, 1 << 45, 4) == 1
    assert _call(lib, 0, 0, 1 << 24, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, big_ld) == 1
    # a large matrix that does fit: 2^20 rows of 2^36 floats (2^58 bytes); C
    # placed 2^50 bytes into A's range overlaps it
    assert _call(lib, 0, 0, 1 << 20, 4, 4, FAKE_A, 1 << 36, FAKE_B, 4, FAKE_A + (1 << 50), 4) == 2


def test_unknown_algo(lib):
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, algo=17) == 1


def test_empty_output_is_a_no_op(lib):
    # M == 0 or N == 0: success without touching the device (even NULL pointers)
    assert _call(lib, 0, 0, 0, 4, 4, 0, 4, 0, 4, 0, 4) == 0
    assert _call(lib, 0, 0, 4, 0, 4, 0, 4, 0, 1, 0, 1) == 0
    assert lib.sgemm_last_launch_count() == 0


def test_degenerate_k_and_alpha_need_no_operands(lib):
    # K == 0 or alpha == 0: A and B may be NULL; only C is needed
    st = _call(lib, 0, 0, 4, 4, 0, 0, 1, 0, 4, FAKE_C, 4, beta=2.0)
    assert st in (0, 3)
    st = _call(lib, 0, 0, 4, 4, 4, 0, 4, 0, 4, FAKE_C, 4, alpha=0.0)
    assert st in (0, 3)


def test_select_algo_is_host_only(lib):
    lib.sgemm_select_algo.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                      ctypes.c_float, ctypes.c_void_p, ctypes.c_int64]
    # 512 x 512 x 384: above the small-product kernel's 2^26 multiply-adds,
    # below the 2^27 from which TMA-ineligible operands are copied aligned
    sel = lambda A, lda, B, ldb, K=384: lib.sgemm_select_algo(0, 0, 512, 512, K, A, lda, B, ldb,
                                                              1.0, 0.0, FAKE_C, 512)
    fa, fb, fc = FAKE_A, FAKE_A + 4 * 512 * 600, FAKE_A + 8 * 512 * 600   # disjoint
    assert sel(fa, 384, fb, 512) == 1                # aligned, ld % 4 == 0 -> TMA
    assert sel(fa + 4, 384, fb, 512) == 2            # A not 16-byte aligned -> cp.async
    assert sel(fa, 385, fb, 512) == 2                # lda % 4 != 0 -> cp.async
    assert sel(fa, 380, fb, 512) == -1               # invalid lda
    # at most 2^26 multiply-adds, K <= 1024 and 608 tiles of 32 x 32: the
    # small-product kernel (512 x 512 is 256 tiles)
    assert sel(fa, 384, fb, 512, K=64) == 6
    big = lambda M, N, K: lib.sgemm_select_algo(0, 0, M, N, K, fa, K, fb, N, 1.0, 0.0, FAKE_C, N)
    assert big(1024, 1024, 64) == 1          # 1024 tiles with a short K: the persistent kernel
    assert big(64, 64, 2048) == 1            # K > 1024: the persistent kernel
    assert big(64, 64, 1024) == 6            # K = 1024, 4 tiles: still the small-product kernel
    assert big(1024, 64, 1024) == 6          # exactly 2^26 multiply-adds, 64 tiles: small
    assert big(1024, 64, 1028) == 1          # just over 2^26 (and K > 1024): persistent
    assert lib.sgemm_select_algo(0, 0, 64, 64, 64, fa, 64, fb, 64, 1.0, 0.0, fc, 64) == 6


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="needs a machine without a GPU")
def test_valid_call_without_gpu_is_unsupported(lib):
    assert _call(lib, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from dense_fp32_matrix_10_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _binding.sgemm_version()


def test_register_split_fits_launch_budget(lib):
    """Every CUDA-core kernel hands registers from its producer warpgroup to its
    math warpgroups with setmaxnreg; the split must not exceed the registers the
    CTA is launched with (ptxas -v of this build), or setmaxnreg.inc would wait
    forever.  The library re-checks this at run time before any launch."""
    from dense_fp32_matrix_10_gb300 import build
    report = build.ptxas_report().splitlines()
    src = open(os.path.join(ROOT, "dense_fp32_matrix_10_gb300", "csrc", "simt_gemm.cuh")).read()
    trans_regs = int(re.search(r"#define SG_SIMT_TRANSPOSER_REGS (\d+)", src).group(1))
    checked = 0
    for i, ln in enumerate(report):
        m = re.search(r"SimtConfigILi(\d+)ELi(\d+)ELb[01]ELb[01]ELi\d+ELi(\d)ELi(\d+)ELb([01])E", ln)
        if not m or "Compiling entry" not in ln:
            continue
        regs = next(int(re.search(r"Used (\d+) registers", x).group(1))
                    for x in report[i + 1:] if "Used" in x)
        math_warps = int(m.group(1)) * int(m.group(2))
        tma, tn, a_trans = m.group(3) == "0", int(m.group(4)), m.group(5) == "1"
        threads = 32 * math_warps + 128
        min_ctas = 1 if math_warps == 8 else 2
        launch = (65536 // (threads * min_ctas)) & ~7
        prod_regs = 24 if (tma and not a_trans) else (trans_regs if a_trans else 40)
        math_regs = min(240, ((threads * launch - 128 * prod_regs) // (32 * math_warps)) & ~7)
        assert regs * threads >= 128 * prod_regs + 32 * math_warps * math_regs, (ln, regs)
        # room for the 8 x TN accumulators, fragments and addresses
        assert math_regs >= (216 if tn == 16 else 168), (ln, math_regs)
        checked += 1
    assert checked >= 8
