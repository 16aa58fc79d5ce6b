"""GPU parity with the oracle on inputs the 3xTF32 split cannot carry.

Two kinds: finite values at the top of the float32 range, whose rounding to
TF32 overflows (every |x| >= (2 - 2^-11) * 2^127), and +-Inf or NaN operands.
The definition (itan.pw "CUDA NVIDIA 4090 高性能計算", 概要; klklkl10086.github.io
"Sgemm单精度矩阵乘法", 问题定义) gives a finite sum for the first kind and
+-Inf or NaN (Inf * 0, Inf - Inf) for the second, and every kernel must give
the oracle's answer: the same NaN positions and infinities, and finite values
bit for bit where the inputs make every product and partial sum exact
(dyadic values, the large ones with 13 significant bits), else within the
per-element bound (K + 2) u S.

The tensor-core kernels reach these results through their NaN repair (a NaN
folded sum is computed again with FP32 FMAs), in the epilogue of a tile one
CTA or cluster covers and in the fixup kernels of shared stream-K tiles
(forced K splits below).
"""
import zlib

import numpy as np
import pytest

import oracle
import sgemm_inputs as si
from gpu_util import U, check_bound, check_exact, dyadic, gpu_sgemm
from test_batched import gpu_batched, oracle_batched
from test_small import _dyadic_stack

pytestmark = pytest.mark.gpu

# 13 and 12 significant bits (products with 6-bit dyadic values stay exact); both round up
# past FLT_MAX as TF32.  TF32_MAX, the largest TF32 value, splits without overflow.
BIG = [(2 - 2.0 ** -12) * 2.0 ** 127, (2 - 2.0 ** -11) * 2.0 ** 127]
TF32_MAX = (2 - 2.0 ** -10) * 2.0 ** 127
FLT_MAX = float(np.finfo(np.float32).max)

# (variant, forced K split): split > 1 shares every tile between CTAs or clusters, so the
# results pass through the fixup kernels
VARIANTS = [("AUTO", 0), ("TC_TF32X3", 0), ("TC_TF32X3", 3), ("TC_PAIR", 0), ("TC_PAIR", 3),
            ("TC_PRESPLIT", 0), ("TC_PRESPLIT", 3), ("TMA_128x128", 0), ("GENERIC", 0)]
IDS = [f"{v}-s{s}" for v, s in VARIANTS]
M, N, K = 300, 264, 256


def stored(op, X):
    """The stored matrix whose op() is the logical X."""
    return np.ascontiguousarray(X.T if op == "T" else X)


def run_both(ta, tb, a, b, c, alpha, beta, variant, split):
    A, B = stored(ta, a), stored(tb, b)
    got = gpu_sgemm(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, c, N, variant=variant,
                    split=split)
    ref, S = oracle.sgemm(ta, tb, A, B, c, alpha, beta, M=M, N=N, K=K, want_bound=True)
    return got, ref, S


def big_operands(rng, side):
    """Logical op(A), op(B): 6-bit dyadic values; on `side`, large entries (one per row of
    op(A) or column of op(B)); the other operand scaled by 2^-20 so every product is finite;
    a zero opposite some large entries (their product is 0, the sum the small terms alone)."""
    a, b = dyadic(rng, M, K), dyadic(rng, K, N)
    placed = []  # (row or column, k, value)
    lines = [0, 5, 127, 128, 255, 256, 299] if side == "A" else [0, 3, 63, 64, 127, 128, 263]
    for i, r in enumerate(lines):
        v = BIG[i % len(BIG)] * (-1.0 if i % 2 else 1.0)
        placed.append((r, (37 * i + 11) % K, v))
    if side == "A":
        b *= np.float32(2.0 ** -20)
        for r, k, v in placed:
            a[r, k] = v
            b[k, (r + 17) % N] = 0.0
    else:
        a *= np.float32(2.0 ** -20)
        for c, k, v in placed:
            b[k, c] = v
            a[(c + 29) % M, k] = 0.0
    return a, b


@pytest.mark.parametrize("side", ["A", "B"])
@pytest.mark.parametrize("ops", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("variant,split", VARIANTS, ids=IDS)
def test_large_finite_inputs_exact(variant, split, ops, side):
    """Entries of (2 - 2^-12) 2^127 and (2 - 2^-11) 2^127 (both signs) times entries
    <= 2^-20: finite products, results equal to the oracle bit for bit."""
    ta, tb = ops
    rng = np.random.default_rng(zlib.crc32(f"{variant}{split}{ops}{side}".encode()))
    a, b = big_operands(rng, side)
    c = dyadic(rng, M, N)
    got, ref, S = run_both(ta, tb, a, b, c, 1.5, -0.5, variant, split)
    assert np.all(np.isfinite(ref))
    check_exact(got, ref, f"{variant} split={split} {ops} large {side}")


@pytest.mark.parametrize("variant,split", VARIANTS, ids=IDS)
def test_flt_max_inputs_within_bound(variant, split):
    """FLT_MAX, -FLT_MAX (24 significant bits: products round) and the largest TF32 value
    against entries <= 2^-20 of random sign: the oracle's finite result within the
    per-element bound."""
    a = si.uniform_pm1(M, K, 92)
    b = (si.uniform_pm1(K, N, 93) * np.float32(2.0 ** -20)).astype(np.float32)
    for r, k, v in ((1, 4, FLT_MAX), (130, 200, -FLT_MAX), (299, 31, TF32_MAX)):
        a[r, k] = v
    c = si.uniform_pm1(M, N, 94)
    got, ref, S = run_both("N", "N", a, b, c, 1.0, 1.0, variant, split)
    assert np.all(np.isfinite(ref)) and np.all(np.isfinite(got)), variant
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.all(err <= (K + 2) * U * S), f"{variant}: worst err/bound {np.max(err / ((K + 2) * U * S)):.3g}"
    check_bound(np.delete(got, [1, 130, 299], 0), np.delete(ref, [1, 130, 299], 0),
                np.delete(S, [1, 130, 299], 0), K, variant)


def inf_nan_operands(rng):
    """Dyadic op(A), op(B) with NaN, +-Inf entries placed to give every IEEE outcome:
    +-Inf rows, Inf * 0 (NaN), Inf - Inf (NaN), an Inf column of op(B), and 0 * Inf."""
    a, b = dyadic(rng, M, K) + np.float32(2.0), np.abs(dyadic(rng, K, N)) + np.float32(0.25)  # a, b > 0
    a[3, 5] = np.nan            # row 3 NaN
    a[7, 9] = np.inf            # row 7 +Inf ...
    b[9, 30] = 0.0              # ... except C[7, 30] = NaN (Inf * 0)
    a[11, 2] = -np.inf          # row 11 -Inf
    a[20, 4] = np.inf           # row 20: Inf - Inf = NaN
    a[20, 6] = -np.inf
    b[40, 100] = np.inf         # column 100 +Inf ...
    a[150, 40] = 0.0            # ... except C[150, 100] = NaN (0 * Inf)
    a[299, 0] = -np.inf         # last row, first k
    b[255, 263] = -np.inf       # last column, last k
    return a, b


@pytest.mark.parametrize("ops", ["NN", "TT"])
@pytest.mark.parametrize("variant,split", VARIANTS, ids=IDS)
def test_inf_nan_operands_match_oracle(variant, split, ops):
    ta, tb = ops
    rng = np.random.default_rng(95)
    a, b = inf_nan_operands(rng)
    c = dyadic(rng, M, N)
    got, ref, _ = run_both(ta, tb, a, b, c, 1.5, -0.5, variant, split)
    assert np.isnan(ref[7, 30]) and np.isnan(ref[20, 0]) and np.isnan(ref[150, 100])
    assert np.isposinf(ref[7, 0]) and np.isneginf(ref[11, 1]) and np.isposinf(ref[0, 100])
    bad = ~((got == ref) | (np.isnan(got) & np.isnan(ref)))
    assert not bad.any(), (f"{variant} split={split} {ops}: {int(bad.sum())} elements differ, first at "
                           f"{tuple(np.argwhere(bad)[0])}")


def test_inf_in_c_with_beta_propagates_and_beta_zero_ignores_it():
    """beta != 0: an Inf in C gives Inf (beta * C); beta == 0: C is not read."""
    rng = np.random.default_rng(96)
    a, b = dyadic(rng, M, K), dyadic(rng, K, N)
    c = dyadic(rng, M, N)
    c[10, 10], c[200, 50] = np.inf, np.nan
    for beta in (-0.5, 0.0):
        got, ref, _ = run_both("N", "N", a, b, c, 1.0, beta, "AUTO", 0)
        assert np.array_equal(got, ref, equal_nan=True), beta


@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_grouped_mode_large_and_inf_inputs(ops):
    """Block-diagonal groups (forced on a short batch): large finite entries and Inf/NaN in
    some products; every product equal to the oracle's (NaN where it has NaN)."""
    ta, tb = ops
    batch, m, n, k = 7, 40, 28, 200
    d = _dyadic_stack(si.make_batched(batch, m, n, k, ta, tb, seed=97, pad=0, gap=4, align=4),
                      np.random.default_rng(98))

    def put_a(p, i, kk, v):  # op(A) of product p, element (i, kk)
        off = p * d["strideA"] + (kk * d["lda"] + i if ta == "T" else i * d["lda"] + kk)
        d["A"][off] = v

    def scale_b(p, f):
        rows = k if tb == "N" else n
        base = p * d["strideB"]
        d["B"][base:base + rows * d["ldb"]] *= np.float32(f)

    scale_b(1, 2.0 ** -20)
    put_a(1, 3, 17, BIG[0])
    put_a(1, 39, 199, -BIG[1])
    put_a(4, 0, 0, np.inf)
    put_a(4, 9, 5, np.nan)
    put_a(6, 20, 100, -np.inf)
    got = gpu_batched(ta, tb, m, n, k, 1.5, -0.5, d, batch, variant="TC_GROUPED")
    ref, _ = oracle_batched(ta, tb, m, n, k, 1.5, -0.5, d, batch)
    bad = ~((got == ref) | (np.isnan(got) & np.isnan(ref)))
    assert not bad.any(), f"grouped {ops}: {int(bad.sum())} elements differ, first at {np.argwhere(bad)[0]}"
