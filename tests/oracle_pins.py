"""Pins that tie the CPU oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
``AssertionError`` when that build disagrees with:

  * the hand-worked examples under ``tests/golden/`` (each cites the definition
    it works out);
  * exact rational arithmetic (``fractions.Fraction``) on tiny inputs;
  * closed forms (identity, all-ones);
  * numpy's int64 matrix product on small-integer inputs (exact);
  * numpy's float64 BLAS product (agreement to double rounding);
  * algebraic invariants (transposition identities, scaling by 2, the
    alpha/beta degenerate cases, padded leading dimensions).

``tests/test_oracle.py`` asserts that the real oracle passes all of them;
``tests/test_oracle_mutants.py`` asserts that each planted mistake in a copy of
the oracle source fails at least one -- so the pins are shown to be able to
catch a dropped term, a wrong sign or index, or a transposed operand.
"""
import glob
import os
from fractions import Fraction

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def load_golden(path):
    """Parse one fixture: op, alpha, beta, A, B, optional C, expect."""
    lines = [ln.split("#", 1)[0].strip() for ln in open(path, encoding="utf-8")]
    lines = [ln for ln in lines if ln]
    out, i = {}, 0
    while i < len(lines):
        tok = lines[i].split()
        key = tok[0]
        if key == "op":
            out["op"] = (tok[1], tok[2])
            i += 1
        elif key in ("alpha", "beta"):
            out[key] = float(tok[1])
            i += 1
        else:
            r, c = int(tok[1]), int(tok[2])
            rows = [[float(v) for v in lines[i + 1 + q].split()] for q in range(r)]
            arr = np.array(rows, dtype=np.float64).reshape(r, c)
            out[key] = arr
            i += 1 + r
    return out


def golden_files():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))


def _opA(A, ta):
    return A.T if ta else A


def exact_product(ta, tb, alpha, A, B, beta, C):
    """Exact rational alpha*op(A)*op(B) + beta*C as a nested list of Fractions."""
    a = _opA(A, ta)
    b = _opA(B, tb)
    M, K = a.shape
    N = b.shape[1]
    fa = [[Fraction(float(a[i, k])) for k in range(K)] for i in range(M)]
    fb = [[Fraction(float(b[k, j])) for j in range(N)] for k in range(K)]
    al, be = Fraction(float(np.float32(alpha))), Fraction(float(np.float32(beta)))
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((fa[i][k] * fb[k][j] for k in range(K)), Fraction(0))
            v = al * s
            if beta != 0:
                v += be * Fraction(float(C[i, j]))
            row.append(v)
        out.append(row)
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _stored(rng, shape, kind):
    if kind == "dyadic":  # multiples of 1/8 in [-8, 8]: every double op on them is exact
        return (rng.integers(-64, 65, size=shape) / 8.0).astype(np.float32)
    if kind == "float":
        return rng.uniform(-1, 1, size=shape).astype(np.float32)
    if kind == "int":
        return rng.integers(-8, 9, size=shape).astype(np.float32)
    raise ValueError(kind)


def _shapes(ta, tb, M, N, K):
    return ((K, M) if ta else (M, K)), ((N, K) if tb else (K, N))


OPS = [(0, 0), (0, 1), (1, 0), (1, 1)]


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------
def pin_golden(orc):
    files = golden_files()
    assert files, "no golden fixtures found"
    for path in files:
        g = load_golden(path)
        ta, tb = (0 if g["op"][0] == "N" else 1), (0 if g["op"][1] == "N" else 1)
        A = g["A"].astype(np.float32)
        B = g["B"].astype(np.float32)
        C = g["C"].astype(np.float32) if "C" in g else None
        R = orc.sgemm_f64(ta, tb, g["alpha"], A, B, g["beta"], C)
        assert np.array_equal(R, g["expect"]), f"{os.path.basename(path)}: {R} != {g['expect']}"


def pin_fraction_dyadic(orc):
    """Dyadic inputs: every intermediate is exact in double, so the oracle must
    equal the exact rational result, for all four op combinations."""
    rng = _rng(11)
    for ta, tb in OPS:
        for (M, N, K) in [(1, 1, 1), (2, 3, 4), (3, 2, 5), (7, 5, 3), (4, 7, 7), (5, 1, 6), (1, 6, 2)]:
            sa, sb = _shapes(ta, tb, M, N, K)
            A, B = _stored(rng, sa, "dyadic"), _stored(rng, sb, "dyadic")
            C = _stored(rng, (M, N), "dyadic")
            for alpha, beta in [(1.0, 0.0), (1.5, 0.5), (-2.0, 1.0), (0.25, -3.0)]:
                R = orc.sgemm_f64(ta, tb, alpha, A, B, beta, C if beta else None)
                X = exact_product(ta, tb, alpha, A, B, beta, C)
                for i in range(M):
                    for j in range(N):
                        assert Fraction(float(R[i, j])) == X[i][j], (ta, tb, M, N, K, i, j)


def pin_fraction_float(orc):
    """General FP32 inputs: the double result is within the recursive-summation
    error bound of the exact rational result, and rounding it to FP32 gives the
    exact result rounded to FP32."""
    rng = _rng(12)
    u = 2.0 ** -53
    for ta, tb in OPS:
        for (M, N, K) in [(3, 4, 7), (6, 5, 2), (2, 2, 6), (5, 7, 7)]:
            sa, sb = _shapes(ta, tb, M, N, K)
            A, B = _stored(rng, sa, "float"), _stored(rng, sb, "float")
            C = _stored(rng, (M, N), "float")
            alpha, beta = 1.25, -0.75
            R = orc.sgemm_f64(ta, tb, alpha, A, B, beta, C)
            X = exact_product(ta, tb, alpha, A, B, beta, C)
            a, b = _opA(A, ta).astype(np.float64), _opA(B, tb).astype(np.float64)
            mag = abs(alpha) * (np.abs(a) @ np.abs(b)) + abs(beta) * np.abs(C.astype(np.float64))
            for i in range(M):
                for j in range(N):
                    err = abs(Fraction(float(R[i, j])) - X[i][j])
                    assert err <= Fraction((K + 3) * u * mag[i, j]), (ta, tb, i, j, float(err))
                    assert np.float32(R[i, j]) == np.float32(float(X[i][j])), (ta, tb, i, j)


def pin_identity(orc):
    """op(A) = I_K (M = K): alpha*op(B) + beta*C exactly."""
    rng = _rng(13)
    for ta, tb in OPS:
        K, N = 9, 6
        A = np.eye(K, dtype=np.float32)
        _, sb = _shapes(ta, tb, K, N, K)
        B = _stored(rng, sb, "float")
        C = _stored(rng, (K, N), "float")
        opb = (B.T if tb else B).astype(np.float64)
        R = orc.sgemm_f64(ta, tb, 1.0, A, B, 0.0, None)
        assert np.array_equal(R, opb), (ta, tb)
        R2 = orc.sgemm_f64(ta, tb, 0.5, A, B, 2.0, C)
        assert np.array_equal(R2, 0.5 * opb + 2.0 * C.astype(np.float64)), (ta, tb)


def pin_all_ones(orc):
    """All-ones A and B: every output is K; with alpha 1.5, beta 0.5, C = 2 it is 1.5K + 1."""
    for ta, tb in OPS:
        for (M, N, K) in [(3, 5, 1), (4, 4, 17), (2, 9, 300)]:
            sa, sb = _shapes(ta, tb, M, N, K)
            A, B = np.ones(sa, np.float32), np.ones(sb, np.float32)
            R = orc.sgemm_f64(ta, tb, 1.0, A, B)
            assert np.all(R == K), (ta, tb, M, N, K)
            C = np.full((M, N), 2.0, np.float32)
            R2 = orc.sgemm_f64(ta, tb, 1.5, A, B, 0.5, C)
            assert np.all(R2 == 1.5 * K + 1), (ta, tb, M, N, K)


def pin_integer_vs_numpy(orc):
    """Small-integer inputs: exact, equal to numpy's int64 matrix product."""
    rng = _rng(14)
    for ta, tb in OPS:
        for (M, N, K) in [(17, 13, 29), (40, 3, 64), (1, 33, 100)]:
            sa, sb = _shapes(ta, tb, M, N, K)
            A, B = _stored(rng, sa, "int"), _stored(rng, sb, "int")
            C = _stored(rng, (M, N), "int")
            ai = (A.T if ta else A).astype(np.int64)
            bi = (B.T if tb else B).astype(np.int64)
            ref = ai @ bi
            R = orc.sgemm_f64(ta, tb, 1.0, A, B)
            assert np.array_equal(R, ref.astype(np.float64)), (ta, tb, M, N, K)
            R2 = orc.sgemm_f64(ta, tb, 2.0, A, B, -1.0, C)
            assert np.array_equal(R2, (2 * ref - C.astype(np.int64)).astype(np.float64)), (ta, tb)


def pin_numpy_float64(orc):
    """Random FP32 inputs: agrees with numpy's float64 BLAS product of the same
    values to within double rounding of the sum (the two sum in different orders)."""
    rng = _rng(15)
    for ta, tb in OPS:
        M, N, K = 37, 29, 211
        sa, sb = _shapes(ta, tb, M, N, K)
        A, B = _stored(rng, sa, "float"), _stored(rng, sb, "float")
        C = _stored(rng, (M, N), "float")
        a = (A.T if ta else A).astype(np.float64)
        b = (B.T if tb else B).astype(np.float64)
        ref = 0.75 * (a @ b) - 1.5 * C.astype(np.float64)
        R = orc.sgemm_f64(ta, tb, 0.75, A, B, -1.5, C)
        bound = 4 * K * 2.0 ** -53 * (0.75 * (np.abs(a) @ np.abs(b)) + 1.5 * np.abs(C))
        assert np.all(np.abs(R - ref) <= bound), (ta, tb)


def pin_transpose_identities(orc):
    """NT(A, B) == NN(A, B^T stored); TN(A, B) == NN(A^T stored, B);
    TT(A, B) == NN(B, A)^T -- bit for bit (same products, same k order)."""
    rng = _rng(16)
    M, N, K = 11, 7, 23
    A = _stored(rng, (M, K), "float")
    Bn = _stored(rng, (K, N), "float")
    Bt = np.ascontiguousarray(Bn.T)
    At = np.ascontiguousarray(A.T)
    nn = orc.sgemm_f64(0, 0, 1.0, A, Bn)
    assert np.array_equal(orc.sgemm_f64(0, 1, 1.0, A, Bt), nn)
    assert np.array_equal(orc.sgemm_f64(1, 0, 1.0, At, Bn), nn)
    assert np.array_equal(orc.sgemm_f64(1, 1, 1.0, At, Bt), nn)
    # TT with independent operands: (op(A) op(B))^T = B^T-stored ... as NN(B, A)
    P = _stored(rng, (K, M), "float")   # stored K x M -> op(P) = P^T is M x K
    Q = _stored(rng, (N, K), "float")   # stored N x K -> op(Q) = Q^T is K x N
    tt = orc.sgemm_f64(1, 1, 1.0, P, Q)
    assert np.array_equal(tt.T, orc.sgemm_f64(0, 0, 1.0, Q, P))


def pin_scaling(orc):
    """With beta = 0, doubling alpha doubles every output exactly; beta*C enters linearly."""
    rng = _rng(17)
    for ta, tb in OPS:
        M, N, K = 9, 14, 33
        sa, sb = _shapes(ta, tb, M, N, K)
        A, B = _stored(rng, sa, "float"), _stored(rng, sb, "float")
        C = _stored(rng, (M, N), "dyadic")
        r1 = orc.sgemm_f64(ta, tb, 0.7, A, B)
        r2 = orc.sgemm_f64(ta, tb, 1.4, A, B)
        assert np.array_equal(r2, 2.0 * r1), (ta, tb)
        # integer-valued product so that adding beta*C stays exact
        Ai, Bi = _stored(rng, sa, "int"), _stored(rng, sb, "int")
        p = orc.sgemm_f64(ta, tb, 1.0, Ai, Bi)
        q = orc.sgemm_f64(ta, tb, 1.0, Ai, Bi, 0.5, C)
        assert np.array_equal(q - p, 0.5 * C.astype(np.float64)), (ta, tb)


def pin_degenerate(orc):
    """beta == 0 never reads C (NaN ignored); alpha == 0 never reads A, B;
    K == 0 gives beta*C."""
    rng = _rng(18)
    M, N, K = 5, 6, 7
    A = _stored(rng, (M, K), "float")
    B = _stored(rng, (K, N), "float")
    Cn = np.full((M, N), np.nan, np.float32)
    C = _stored(rng, (M, N), "dyadic")
    R = orc.sgemm_f64(0, 0, 1.0, A, B, 0.0, Cn)
    assert np.all(np.isfinite(R))
    An = np.full((M, K), np.nan, np.float32)
    R0 = orc.sgemm_f64(0, 0, 0.0, An, B, 0.5, C)
    assert np.array_equal(R0, 0.5 * C.astype(np.float64))
    Z = orc.sgemm_f64(0, 0, 0.0, An, B, 0.0, Cn)
    assert np.array_equal(Z, np.zeros((M, N)))
    Ak = np.zeros((M, 0), np.float32)
    Bk = np.zeros((0, N), np.float32)
    Rk = orc.sgemm_f64(0, 0, 3.0, Ak, Bk, -2.0, C)
    assert np.array_equal(Rk, -2.0 * C.astype(np.float64))


def pin_padded_ld(orc):
    """Padded leading dimensions: NaN in the padding columns never reaches a result,
    and the result equals the unpadded one."""
    rng = _rng(19)
    for ta, tb in OPS:
        M, N, K = 6, 5, 9
        sa, sb = _shapes(ta, tb, M, N, K)
        A, B = _stored(rng, sa, "float"), _stored(rng, sb, "float")
        C = _stored(rng, (M, N), "float")
        def pad(x, extra):
            big = np.full((x.shape[0], x.shape[1] + extra), np.nan, np.float32)
            big[:, : x.shape[1]] = x
            return big[:, : x.shape[1]]
        ref = orc.sgemm_f64(ta, tb, 1.5, A, B, 0.5, C)
        got = orc.sgemm_f64(ta, tb, 1.5, pad(A, 3), pad(B, 5), 0.5, pad(C, 2))
        assert np.array_equal(got, ref), (ta, tb)


def pin_entries_match_full(orc):
    """The per-entry routine equals the full product bit for bit."""
    rng = _rng(20)
    for ta, tb in OPS:
        M, N, K = 13, 10, 27
        sa, sb = _shapes(ta, tb, M, N, K)
        A, B = _stored(rng, sa, "float"), _stored(rng, sb, "float")
        C = _stored(rng, (M, N), "float")
        full = orc.sgemm_f64(ta, tb, -1.25, A, B, 0.5, C)
        I = rng.integers(0, M, size=40)
        J = rng.integers(0, N, size=40)
        ent = orc.sgemm_entries_f64(ta, tb, -1.25, A, B, 0.5, C, I, J)
        assert np.array_equal(ent, full[I, J]), (ta, tb)
        # and against exact arithmetic on one entry, independently of the full routine
        X = exact_product(ta, tb, -1.25, A, B, 0.5, C)
        assert np.float32(ent[0]) == np.float32(float(X[I[0]][J[0]]))


def pin_threads_invariant(orc):
    """Splitting rows over threads changes no bit."""
    rng = _rng(21)
    A = _stored(rng, (53, 41), "float")
    B = _stored(rng, (41, 19), "float")
    r1 = orc.sgemm_f64(0, 0, 1.0, A, B, threads=1)
    r7 = orc.sgemm_f64(0, 0, 1.0, A, B, threads=7)
    assert np.array_equal(r1, r7)


# ------------------------------------------------------------ transpose
TRANSPOSE_GOLDEN_DIR = os.path.join(GOLDEN_DIR, "transpose")


def _bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def pin_transpose_golden(orc):
    files = sorted(glob.glob(os.path.join(TRANSPOSE_GOLDEN_DIR, "*.txt")))
    assert len(files) >= 2
    for f in files:
        g = load_golden(f)
        X = g["in"].astype(np.float32)
        out = orc.transpose_f32(X)
        assert np.array_equal(_bits(out), _bits(g["expect"])), os.path.basename(f)


def pin_transpose_numpy_and_involution(orc):
    """Bit-exact equal to numpy's own transpose (NaN payloads, signed zeros,
    infinities and subnormals included) on ragged shapes, and transposing
    twice gives the input back."""
    rng = _rng(41)
    for rows, cols in [(1, 1), (1, 7), (7, 1), (5, 3), (33, 17), (64, 130)]:
        X = rng.standard_normal((rows, cols)).astype(np.float32)
        flat = X.reshape(-1)
        flat[:: 5] = np.float32(-0.0)
        flat[1:: 7] = np.float32(np.inf)
        flat[2:: 11] = np.float32(1e-42)            # subnormal
        bits = flat.view(np.uint32)
        bits[3:: 13] = 0x7FC0ABCD                   # NaN with a payload
        T = orc.transpose_f32(X)
        assert np.array_equal(_bits(T), _bits(X.T)), (rows, cols)
        assert np.array_equal(_bits(orc.transpose_f32(T)), _bits(X)), (rows, cols)


def pin_transpose_leading_dimensions(orc):
    """Padded input rows are not read and padded output rows not written."""
    rng = _rng(42)
    rows, cols = 9, 6
    big_in = np.full((rows, cols + 3), np.nan, np.float32)
    big_in[:, :cols] = _stored(rng, (rows, cols), "dyadic")
    big_out = np.full((cols, rows + 5), 7.0, np.float32)
    orc.transpose_f32(big_in[:, :cols], out=big_out[:, :rows])
    assert np.array_equal(big_out[:, :rows], big_in[:, :cols].T)
    assert np.all(big_out[:, rows:] == 7.0)


# ------------------------------------------------------------ strided batch
def _strided_view(flat, batch, rows, cols, ld, stride):
    """numpy's own view of the strided-batch layout: element (b, r, c) at
    flat[b*stride + r*ld + c]."""
    return np.lib.stride_tricks.as_strided(flat, shape=(batch, rows, cols),
                                           strides=(4 * stride, 4 * ld, 4), writeable=False)


def pin_batched_closed_form(orc):
    """A_b = (b+1) * I (square, K = M): product b is exactly (b+1) * op(B_b);
    with transB the transposed B_b, so a swapped stride or op shows."""
    M = K = 6
    N, batch = 5, 4
    rng = _rng(31)
    eye = np.eye(M, dtype=np.float32)
    A = np.concatenate([(b + 1) * eye.ravel() for b in range(batch)]).astype(np.float32)
    for tb in (0, 1):
        rows, cols = (N, K) if tb else (K, N)
        B = _stored(rng, (batch * rows * cols,), "int")
        R = orc.sgemm_strided_batched_f64(0, tb, M, N, K, 1.0, A, M, M * M, B, cols, rows * cols,
                                          0.0, None, N, M * N, batch)
        Bv = _strided_view(B, batch, rows, cols, cols, rows * cols)
        for b in range(batch):
            Bb = Bv[b].T if tb else Bv[b]
            assert np.array_equal(R[b], (b + 1) * Bb.astype(np.float64)), (tb, b)


def pin_batched_broadcast_and_interleaved(orc):
    """Head-interleaved inputs (lda = heads * K, strideA = K: the packed Q K^T
    layout of attention) and a shared operand (strideB = 0), against numpy's
    float64 matmul on numpy's own strided views; integer data, so exact."""
    heads, M, N, K = 3, 5, 4, 7
    rng = _rng(32)
    A = _stored(rng, (M * heads * K,), "int")
    B = _stored(rng, (K * N,), "int")
    C = _stored(rng, (heads * M * N,), "int")
    R = orc.sgemm_strided_batched_f64(0, 0, M, N, K, 2.0, A, heads * K, K, B, N, 0, -1.0, C, N,
                                      M * N, heads)
    Av = _strided_view(A, heads, M, K, heads * K, K).astype(np.float64)
    Bv = _strided_view(B, heads, K, N, N, 0).astype(np.float64)
    Cv = _strided_view(C, heads, M, N, N, M * N).astype(np.float64)
    assert np.array_equal(R, 2.0 * np.matmul(Av, Bv) - Cv)
    # transposed A read from the same interleaved buffer (op(A) = A_b^T: K x M stored)
    At = _stored(rng, (K * heads * M,), "int")
    R = orc.sgemm_strided_batched_f64(1, 0, M, N, K, 1.0, At, heads * M, M, B, N, 0, 0.0, None, N,
                                      M * N, heads)
    Atv = _strided_view(At, heads, K, M, heads * M, M).astype(np.float64)
    assert np.array_equal(R, np.matmul(np.swapaxes(Atv, 1, 2), Bv))


def pin_batched_gaps_unread(orc):
    """Elements between the matrices of a padded batch (NaN here) are never
    read, and beta == 0 reads no C at all."""
    batch, M, N, K = 3, 4, 3, 5
    rng = _rng(33)
    sa, sb = M * K + 9, K * N + 2
    A = np.full(batch * sa, np.nan, np.float32)
    B = np.full(batch * sb, np.nan, np.float32)
    for b in range(batch):
        A[b * sa: b * sa + M * K] = _stored(rng, (M * K,), "dyadic")
        B[b * sb: b * sb + K * N] = _stored(rng, (K * N,), "dyadic")
    C = np.full(batch * M * N, np.nan, np.float32)
    R = orc.sgemm_strided_batched_f64(0, 0, M, N, K, 1.0, A, K, sa, B, N, sb, 0.0, C, N, M * N, batch)
    assert np.all(np.isfinite(R))
    Av = _strided_view(A, batch, M, K, K, sa).astype(np.float64)
    Bv = _strided_view(B, batch, K, N, N, sb).astype(np.float64)
    assert np.array_equal(R, np.matmul(Av, Bv))


ALL_PINS = [
    pin_golden, pin_fraction_dyadic, pin_fraction_float, pin_identity, pin_all_ones,
    pin_integer_vs_numpy, pin_numpy_float64, pin_transpose_identities, pin_scaling,
    pin_degenerate, pin_padded_ld, pin_entries_match_full, pin_threads_invariant,
    pin_batched_closed_form, pin_batched_broadcast_and_interleaved, pin_batched_gaps_unread,
    pin_transpose_golden, pin_transpose_numpy_and_involution, pin_transpose_leading_dimensions,
]
