"""Seeded synthetic inputs and the workload table for row-major SGEMM.

This module is shared by the tests and the benchmark.  It holds no GEMM
arithmetic: only random number generation, the pages' integer fill pattern,
padding of stored matrices, the configuration table, and the FLOP / byte
counts used to turn times into rates.

Sources:
  * uniform[-1, 1) fill ``2*u - 1`` and the integer fill ``(j - i) % 3`` with C
    truncating modulo: klklkl10086.github.io "Sgemm单精度矩阵乘法", 代码框架
    (random_matrix).  The page's drand48 is unseeded; here u comes from numpy's
    PCG64 with a fixed seed, so runs are reproducible.
  * FLOP count 2*M*N*K: same page, 问题定义; itan.pw "CUDA NVIDIA 4090
    高性能計算", §2.1.
  * Minimum bytes: A and B read once, C written once, and C read when
    beta != 0 (§2.1 of the itan.pw page prints (MK+KN+2MN)*4 but evaluates
    3*1024^2*4; the beta-dependent reading is used).
  * The configurations: the workload table of the benchmark contract
    (1000x1300x700 problem of the page's 代码框架, the 1024^3 base size of
    §2.1, the 4096^3 example of 问题定义, a transpose sweep, ragged padded
    shapes, and fully connected layer shapes, 概要).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "uniform_pm1", "normal", "int_pattern", "stored_shape", "embed_padded",
    "Case", "CASES", "case", "make_case", "flops", "min_bytes", "HEADLINE",
    "embed_batched", "make_batched", "BatchedCase", "BATCHED_CASES", "batched_case",
]


def _rng(seed, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def uniform_pm1(rows: int, cols: int, seed: int, stream: int = 0) -> np.ndarray:
    """float32 matrix of 2u - 1 with u ~ U[0, 1) in float64, then rounded to float32."""
    u = _rng(seed, stream).random((rows, cols), dtype=np.float64)
    return (2.0 * u - 1.0).astype(np.float32)


def normal(rows: int, cols: int, seed: int, stream: int = 0, std: float = 1.0) -> np.ndarray:
    """float32 matrix of N(0, std^2) samples (float64 draw, rounded to float32)."""
    z = _rng(seed, stream).standard_normal((rows, cols), dtype=np.float64)
    return (z * std).astype(np.float32)


def int_pattern(rows: int, cols: int) -> np.ndarray:
    """A(i, j) = (j - i) % 3 with C semantics (truncation toward zero): values in {-2..2}.

    Computed on int64, so a zero is +0.0 after the cast, as the page's int->float
    conversion gives.
    """
    i = np.arange(rows, dtype=np.int64)[:, None]
    j = np.arange(cols, dtype=np.int64)[None, :]
    return np.fmod(j - i, 3).astype(np.float32)


def stored_shape(op: str, rows: int, cols: int) -> tuple[int, int]:
    """Shape of the stored matrix whose op() is rows x cols."""
    return (cols, rows) if op.upper() in ("T", "C") else (rows, cols)


def embed_padded(X: np.ndarray, ld: int, fill: float = float("nan")) -> np.ndarray:
    """Copy X (rows x cols) into a rows x ld buffer; the padding columns hold ``fill``.

    Returns the full padded array; ``result[:, :cols]`` is the logical matrix.
    NaN padding makes any read of a padding element visible in the result.
    """
    rows, cols = X.shape
    if ld < cols:
        raise ValueError("ld < cols")
    out = np.full((rows, ld), fill, dtype=np.float32)
    out[:, :cols] = X
    return out


@dataclasses.dataclass(frozen=True)
class Case:
    """One SGEMM workload: C = alpha * op(A) * op(B) + beta * C, row-major."""
    name: str
    M: int
    N: int
    K: int
    transA: str = "N"
    transB: str = "N"
    alpha: float = 1.0
    beta: float = 0.0
    seed: int = 0
    dist: str = "uniform"          # "uniform" | "int" | "fc"
    pad: int = 0                   # extra floats per stored row of A, B and C
    c_init: str = "zero"           # "zero" | "uniform"
    group: str = ""

    @property
    def ops(self) -> str:
        return self.transA + self.transB


def _transpose_sweep(M, N, K, seed, pad, group):
    return [Case(f"{group}_{ta}{tb}", M, N, K, ta, tb, 1.0, 1.0, seed, "uniform", pad, "uniform", group)
            for ta in "NT" for tb in "NT"]


CASES: list[Case] = [
    # 1: the page's own test problem (non tile-multiple), random and integer fills
    Case("pr1_random", 1000, 1300, 700, seed=1, group="pr1"),
    Case("pr1_int", 1000, 1300, 700, seed=1, dist="int", group="pr1"),
    # 2: the pages' base size
    Case("square1024", 1024, 1024, 1024, seed=2, group="square1024"),
    # 3: headline
    Case("square4096", 4096, 4096, 4096, alpha=1.5, beta=-0.5, seed=3, c_init="uniform", group="square4096"),
    # 4: transpose sweep at 2048^3 and ragged padded shapes
    *_transpose_sweep(2048, 2048, 2048, 4, 0, "t2048"),
    *_transpose_sweep(4097, 3001, 2053, 5, 7, "ragged"),
    # 5: fully connected layer shapes: activations N(0,1), weights N(0,1/K)
    Case("fc_8192x4096x1024", 8192, 4096, 1024, seed=6, dist="fc", group="fc"),
    Case("fc_16384x1024x4096", 16384, 1024, 4096, seed=7, dist="fc", group="fc"),
    Case("skinny_64x4096x16384", 64, 4096, 16384, seed=8, dist="fc", group="fc"),
    # beyond the five configurations: the ragged shape with every stored row padded by one float,
    # so no leading dimension is a multiple of 4 (operands TMA cannot load directly)
    Case("unaligned_4097x3001x2053", 4097, 3001, 2053, "N", "N", 1.0, 1.0, 9, "uniform", 1, "uniform",
         "unaligned"),
]

HEADLINE = "square4096"


def case(name: str) -> Case:
    for c in CASES:
        if c.name == name:
            return c
    raise KeyError(name)


def make_case(c: Case, rows_a: int | None = None):
    """Generate the stored operands of a case.

    Returns dict(A, B, C, lda, ldb, ldc) of float32 numpy arrays; with
    ``pad > 0`` each array is the full padded buffer (rows x ld) and its padding
    holds NaN.  A and B are generated on their STORED index space (so the
    integer pattern follows the stored (row, col) of each matrix, as the page's
    random_matrix does for A and B).
    """
    a_shape = stored_shape(c.transA, c.M, c.K)
    b_shape = stored_shape(c.transB, c.K, c.N)
    if c.dist == "uniform":
        A = uniform_pm1(*a_shape, c.seed, 1)
        B = uniform_pm1(*b_shape, c.seed, 2)
    elif c.dist == "int":
        A = int_pattern(*a_shape)
        B = int_pattern(*b_shape)
    elif c.dist == "fc":
        A = normal(*a_shape, c.seed, 1, 1.0)
        B = normal(*b_shape, c.seed, 2, 1.0 / math.sqrt(c.K))
    else:
        raise ValueError(c.dist)
    if c.c_init == "uniform":
        C = uniform_pm1(c.M, c.N, c.seed, 3)
    else:
        C = np.zeros((c.M, c.N), dtype=np.float32)
    out = {}
    for name, X in (("A", A), ("B", B), ("C", C)):
        ld = X.shape[1] + c.pad
        out[name] = embed_padded(X, ld) if c.pad else X
        out["ld" + name.lower()] = ld
    return out


def embed_batched(X: np.ndarray, ld: int, stride: int, fill: float = float("nan")) -> np.ndarray:
    """Lay out a (batch, rows, cols) stack as a flat buffer: matrix b starts at
    b*stride, rows ld apart; padding and gaps hold ``fill``.  stride 0 stores
    the single matrix X[0] (one matrix shared by every product)."""
    batch, rows, cols = X.shape
    if ld < cols:
        raise ValueError("ld < cols")
    if stride == 0:
        out = np.full(rows * ld, fill, dtype=np.float32)
        out.reshape(rows, ld)[:, :cols] = X[0]
        return out
    if stride < rows * ld:
        raise ValueError("stride smaller than one matrix")
    out = np.full(max(batch - 1, 0) * stride + rows * ld, fill, dtype=np.float32)
    for b in range(batch):
        out[b * stride:b * stride + rows * ld].reshape(rows, ld)[:, :cols] = X[b]
    return out


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def make_batched(batch: int, M: int, N: int, K: int, transA: str = "N", transB: str = "N", seed: int = 0,
                 dist: str = "uniform", pad: int = 0, gap: int = 0, align: int = 4, shared: str = "",
                 c_init: str = "uniform"):
    """Operands of a strided batch of ``batch`` products, as flat float32 buffers.

    Each stored matrix has ``pad`` extra floats per row; consecutive matrices
    are ``rows*ld + gap`` floats apart, rounded up to a multiple of ``align``
    (align=4 keeps every matrix 16-byte aligned).  ``shared`` may name "A"
    and/or "B": that operand is one matrix with stride 0.  Padding and gaps
    hold NaN, so a read of them poisons a result and a write to them shows.
    Returns dict(A, B, C, lda, ldb, ldc, strideA, strideB, strideC, stacks)
    where ``stacks`` holds the (batch, rows, cols) logical matrices.
    """
    a_shape = stored_shape(transA, M, K)
    b_shape = stored_shape(transB, K, N)
    nA = 1 if "A" in shared else batch
    nB = 1 if "B" in shared else batch
    if dist == "uniform":
        A = uniform_pm1(nA * a_shape[0], a_shape[1], seed, 1)
        B = uniform_pm1(nB * b_shape[0], b_shape[1], seed, 2)
    elif dist == "fc":
        A = normal(nA * a_shape[0], a_shape[1], seed, 1, 1.0)
        B = normal(nB * b_shape[0], b_shape[1], seed, 2, 1.0 / math.sqrt(max(K, 1)))
    else:
        raise ValueError(dist)
    A = A.reshape(nA, *a_shape)
    B = B.reshape(nB, *b_shape)
    if c_init == "uniform":
        C = uniform_pm1(batch * M, N, seed, 3).reshape(batch, M, N)
    else:
        C = np.zeros((batch, M, N), dtype=np.float32)
    out = {"stacks": {"A": A, "B": B, "C": C}}
    for name, X, is_shared in (("A", A, "A" in shared), ("B", B, "B" in shared), ("C", C, False)):
        rows, cols = X.shape[1:]
        ld = cols + pad
        stride = 0 if is_shared else _round_up(rows * ld + gap, align)
        out[name] = embed_batched(X, ld, stride)
        out["ld" + name.lower()] = ld
        out["stride" + name] = stride
    return out


@dataclasses.dataclass(frozen=True)
class BatchedCase:
    """A strided batch of identical-shape products C_b = alpha op(A_b) op(B_b) + beta C_b."""
    name: str
    batch: int
    M: int
    N: int
    K: int
    transA: str = "N"
    transB: str = "N"
    alpha: float = 1.0
    beta: float = 0.0
    seed: int = 0
    dist: str = "fc"
    shared: str = ""

    @property
    def ops(self) -> str:
        return self.transA + self.transB


BATCHED_CASES: list[BatchedCase] = [
    # many fully connected layers of one network size per call (itan.pw page, 概要)
    BatchedCase("batched_fc_64x512x1024x1024", 64, 512, 1024, 1024, seed=21),
    # one weight matrix shared by every product (stride 0 for B)
    BatchedCase("batched_fc_shared_w_32x2048x1024x1024", 32, 2048, 1024, 1024, seed=22, shared="B"),
    # many small products: the launch and tail overheads dominate
    BatchedCase("batched_small_8192x64x64x64", 8192, 64, 64, 64, seed=23, dist="uniform"),
    # small outputs, long K: two products to a tensor-core tile
    BatchedCase("batched_small_k1024_2048x64x64x1024", 2048, 64, 64, 1024, seed=24, dist="uniform"),
    # tiny products: four to a tensor-core tile
    BatchedCase("batched_tiny_16384x32x32x32", 16384, 32, 32, 32, seed=25, dist="uniform"),
]


def batched_case(name: str) -> BatchedCase:
    for c in BATCHED_CASES:
        if c.name == name:
            return c
    raise KeyError(name)


def flops(M: int, N: int, K: int) -> int:
    """Floating point operations of one SGEMM: one multiply and one add per term, 2*M*N*K."""
    return 2 * int(M) * int(N) * int(K)


def min_bytes(M: int, N: int, K: int, beta: float) -> int:
    """Algorithmic minimum DRAM bytes: read A and B once, write C, read C if beta != 0."""
    c_passes = 2 if beta != 0.0 else 1
    return 4 * (int(M) * int(K) + int(K) * int(N) + c_passes * int(M) * int(N))
