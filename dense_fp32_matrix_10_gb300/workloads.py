"""Seeded synthetic inputs for single-precision GEMM workloads.

This module only draws numbers and names shapes; it performs none of the GEMM
arithmetic, so both the GPU tests/bench and the CPU oracle can take their inputs
from it without sharing any computation.

Recipe (the pages fix the shapes and value distributions, not a generator):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed;
  * A, then B, then C are drawn in that order, each in its *stored* layout
    (for op(B) = T, B is drawn as an N x K array);
  * ``uniform``  -> ``torch.rand(...) * 2 - 1`` (i.i.d. uniform on [-1, 1));
    ``normal``   -> ``torch.randn(...)`` (i.i.d. standard normal);
    ``int``      -> integers drawn uniformly from [-8, 8] (exact in FP32 and in
    TF32; used for the bit-exact checks).
  * C is drawn only when beta != 0; otherwise it is zero-initialised.

The shapes, seeds and scalars below restate the workloads of the pages: square
products of 256 ... 4096 (the RTX 3060 1024^2 case and the RTX 3090 512..4096
table of "GPU矩阵乘法优化：共享内存Tiling技术实战" section 5), the transposed-B
form D = alpha*A*B^T + beta*C of the cloud.baidu.com naive-vs-2D-tiling article,
and three ragged / skinny shapes with odd leading dimensions.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import torch


@dataclass(frozen=True)
class Case:
    name: str
    M: int
    N: int
    K: int
    transA: int
    transB: int
    dist: str
    seed: int
    alpha: float
    beta: float

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def a_shape(self) -> Tuple[int, int]:
        return (self.K, self.M) if self.transA else (self.M, self.K)

    def b_shape(self) -> Tuple[int, int]:
        return (self.N, self.K) if self.transB else (self.K, self.N)

    def as_int(self) -> "Case":
        """The same shape/op/scalars with integer-valued inputs (seed + 100)."""
        return Case(self.name + "_int", self.M, self.N, self.K, self.transA, self.transB,
                    "int", self.seed + 100, self.alpha, self.beta)


def _draw(shape, dist: str, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-8, 9, shape, generator=g, dtype=torch.int32).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(case: Case):
    """(A, B, C) as contiguous CPU float32 tensors in stored layout."""
    g = torch.Generator("cpu").manual_seed(case.seed)
    A = _draw(case.a_shape(), case.dist, g)
    B = _draw(case.b_shape(), case.dist, g)
    if case.beta != 0.0:
        C = _draw((case.M, case.N), case.dist, g)
    else:
        C = torch.zeros((case.M, case.N), dtype=torch.float32)
    return A, B, C


def make_matrix(shape, dist: str, seed: int) -> torch.Tensor:
    """One seeded matrix (used by the shape sweeps of the tests)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return _draw(tuple(shape), dist, g)


# The five workload families.  Family 0 is the small case the oracle finishes
# in well under a second; family 2's 4096^3 case is the headline throughput
# workload.
SMALL_256 = Case("nn_256_uniform_s0", 256, 256, 256, 0, 0, "uniform", 0, 1.0, 0.0)
SQUARE_1024 = Case("nn_1024_uniform_s1", 1024, 1024, 1024, 0, 0, "uniform", 1, 1.0, 0.0)
SWEEP = [Case(f"nn_{n}_normal_s2", n, n, n, 0, 0, "normal", 2, 1.0, 0.0)
         for n in (512, 1024, 2048, 4096)]
NT_4096 = Case("nt_4096_uniform_s3", 4096, 4096, 4096, 0, 1, "uniform", 3, 1.5, 0.5)
RAGGED = [Case("nn_1000x1013x997_uniform_s4", 1000, 1013, 997, 0, 0, "uniform", 4, 1.0, 1.0),
          Case("nn_8192x64x4096_uniform_s4", 8192, 64, 4096, 0, 0, "uniform", 4, 1.0, 1.0),
          Case("nn_65x4097x129_uniform_s4", 65, 4097, 129, 0, 0, "uniform", 4, 1.0, 1.0)]
HEADLINE = SWEEP[-1]

ALL_CASES: List[Case] = [SMALL_256, SQUARE_1024, *SWEEP, NT_4096, *RAGGED]
