"""Plant mistakes in copies of the oracle source and check the pins catch each.

Every mutant is a plausible slip (a transposed operand, a dropped or doubled
term, a wrong sign, an off-by-one in k, a wrong leading dimension, a single
precision accumulator).  Each is compiled from a temporary copy of
``oracle/oracle_sgemm.c`` on the CPU and run against ``tests/oracle_pins.py`` in
a child process (a crash counts as caught).  The committed oracle is never
modified.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_sgemm.c")

# (id, text to replace, replacement)
MUTANTS = [
    ("opA_index_swapped",
     "return transA ? (double)A[k * lda + i] : (double)A[i * lda + k];",
     "return transA ? (double)A[i * lda + k] : (double)A[k * lda + i];"),
    ("opB_index_swapped",
     "return transB ? (double)B[j * ldb + k] : (double)B[k * ldb + j];",
     "return transB ? (double)B[k * ldb + j] : (double)B[j * ldb + k];"),
    ("beta_term_dropped",
     "r[j] += job->beta * (double)crow[j];",
     "r[j] += 0.0 * (double)crow[j];"),
    ("beta_used_as_alpha",
     "r[j] += job->beta * (double)crow[j];",
     "r[j] += job->alpha * (double)crow[j];"),
    ("C_read_when_beta_zero",
     "if (job->beta != 0.0) {",
     "if (job->C != NULL) {"),
    ("alpha_dropped_ikj",
     "r[j] = job->alpha * acc[j];",
     "r[j] = acc[j];"),
    ("alpha_dropped_ijk",
     "r[j] = job->alpha * s;",
     "r[j] = s;"),
    ("last_k_dropped_ikj",
     "for (int64_t k = 0; k < K; ++k) {\n        const double a",
     "for (int64_t k = 0; k < K - 1; ++k) {\n        const double a"),
    ("first_k_dropped_ijk",
     "for (int64_t k = 0; k < K; ++k)\n          s += op_a(job->A",
     "for (int64_t k = 1; k < K; ++k)\n          s += op_a(job->A"),
    ("sign_flipped",
     "acc[j] += a * (double)brow[j];",
     "acc[j] -= a * (double)brow[j];"),
    ("single_precision_accumulator",
     "for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)brow[j];",
     "for (int64_t j = 0; j < N; ++j) acc[j] = (double)(float)(acc[j] + a * (double)brow[j]);"),
    ("ldc_taken_as_N",
     "const float *crow = job->C + i * job->ldc;",
     "const float *crow = job->C + i * job->N;"),
    ("ldb_taken_as_N",
     "const float *brow = job->B + k * job->ldb;",
     "const float *brow = job->B + k * job->N;"),
    ("opA_ignores_trans_in_dot",
     "s += op_a(job->A, job->lda, job->transA, i, k) * op_b(job->B, job->ldb, 1, k, j);",
     "s += op_a(job->A, job->lda, 0, i, k) * op_b(job->B, job->ldb, 1, k, j);"),
    ("entries_ignore_transB",
     "s += op_a(A, lda, transA, i, k) * op_b(B, ldb, transB, k, j);",
     "s += op_a(A, lda, transA, i, k) * op_b(B, ldb, 0, k, j);"),
    ("entries_drop_beta",
     "if (beta != 0.0f) r += (double)beta * (double)C[i * ldc + j];",
     "(void)ldc;"),
    ("transpose_copies_instead",
     "out[c * ld_out + r] = in[r * ld_in + c];",
     "out[r * ld_out + c] = in[r * ld_in + c];"),
    ("transpose_uses_ld_in_for_out",
     "out[c * ld_out + r] = in[r * ld_in + c];",
     "out[c * ld_in + r] = in[r * ld_in + c];"),
    ("transpose_last_column_dropped",
     "for (int64_t c = 0; c < cols; ++c) out[c * ld_out + r]",
     "for (int64_t c = 0; c + 1 < cols; ++c) out[c * ld_out + r]"),
    ("row_block_short_by_one",
     "j->row_end = j->row_begin + per < M ? j->row_begin + per : M;",
     "j->row_end = j->row_begin + per - 1 < M ? j->row_begin + per - 1 : M;"),
]

RUNNER = r"""
import sys
sys.path.insert(0, {root!r})
from oracle import Oracle
from tests.oracle_pins import ALL_PINS
o = Oracle({lib!r})
failed = []
for p in ALL_PINS:
    try:
        p(o)
    except Exception as e:  # AssertionError or a rejected call
        failed.append(p.__name__)
print("FAILED:" + ",".join(failed))
"""


def test_mutant_table_anchors_exist():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"{name}: anchor found {src.count(old)} times"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    sys.path.insert(0, ROOT)
    from oracle import build as obuild
    src = open(SRC).read()
    assert src.count(old) == 1
    msrc = tmp_path / "oracle_mutant.c"
    msrc.write_text(src.replace(old, new))
    lib = str(tmp_path / "liboracle_mutant.so")
    obuild.build(force=True, src=str(msrc), out=lib)
    proc = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, lib=lib)],
                          capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        return  # crashed or raised outside a pin: caught
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("FAILED:")][-1]
    failed = [f for f in line[len("FAILED:"):].split(",") if f]
    assert failed, f"mutant {name} passed every pin"
