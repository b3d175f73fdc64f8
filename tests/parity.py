"""Helpers of the GPU parity tests: run the library on seeded inputs and
compare element by element with the CPU oracle.

Tolerance (random inputs of unit scale):
    ||G - R||_F / ||R||_F <= 1e-5   and   max |G - R| <= 1e-4 * sqrt(K)
with G the GPU result and R the FP64-accumulated oracle result; bit-exact
(G == R) on integer-valued inputs, where every partial sum is an integer below
2^24 and so exact in FP32 in any summation order.
"""
import math

import numpy as np
import torch

REL_FRO = 1e-5
ABS_PER_SQRT_K = 1e-4


def tolerance_report(G, R, K):
    G = np.asarray(G, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    diff = G - R
    nr = np.linalg.norm(R)
    rel = float(np.linalg.norm(diff) / nr) if nr > 0 else float(np.linalg.norm(diff))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    return rel, mx


def assert_close(G, R, K, what=""):
    rel, mx = tolerance_report(G, R, K)
    lim = ABS_PER_SQRT_K * math.sqrt(max(K, 1))
    assert np.all(np.isfinite(G)), f"{what}: non-finite output"
    assert rel <= REL_FRO and mx <= lim, f"{what}: rel_fro={rel:.3e} max_abs={mx:.3e} (lim {lim:.3e})"
    return rel, mx


def assert_bit_exact(G, R, what=""):
    G = np.asarray(G, dtype=np.float64)
    bad = np.flatnonzero(G != R)
    assert bad.size == 0, f"{what}: {bad.size} outputs differ, first at flat {bad[:5]}: " \
                          f"{G.flat[bad[:5]]} vs {np.asarray(R).flat[bad[:5]]}"


def padded(t: torch.Tensor, extra_cols: int, fill=float("nan")):
    """A row-major view of `t` whose rows are `extra_cols` longer (ld > cols);
    the padding holds `fill`."""
    r, c = t.shape
    big = torch.full((r, c + extra_cols), fill, dtype=t.dtype, device=t.device)
    big[:, :c] = t
    return big[:, :c]


def offset_view(t: torch.Tensor, elems: int):
    """A copy of `t` placed `elems` floats past a 16-byte boundary (misaligned
    base pointer), same ld."""
    r, c = t.shape
    flat = torch.empty(r * c + elems + 4, dtype=t.dtype, device=t.device)
    v = flat[elems: elems + r * c].view(r, c)
    v.copy_(t)
    return v


def sample_indices(M, N, n, seed):
    """n sampled (i, j) plus the four corners and the last row/column edges."""
    rng = np.random.default_rng(seed)
    I = list(rng.integers(0, M, size=n))
    J = list(rng.integers(0, N, size=n))
    for i, j in [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]:
        I.append(i)
        J.append(j)
    for j in rng.integers(0, N, size=min(N, 64)):
        I.append(M - 1)
        J.append(int(j))
    for i in rng.integers(0, M, size=min(M, 64)):
        I.append(int(i))
        J.append(N - 1)
    return np.array(I, dtype=np.int64), np.array(J, dtype=np.int64)
