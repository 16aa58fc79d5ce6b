"""GPU parity of the 3xTF32 tensor-core kernel (variant TC_TF32X3), every operand layout.

Dyadic inputs (multiples of 2^-6) split exactly (lo = 0) and all partial sums
are exact, so those results must equal the oracle bit for bit: this checks
the operand layouts, swizzles, descriptors, the TMEM A operand, the K split
and the epilogue.  Random inputs must meet the same per-element and
Frobenius bounds as every other path.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

V = "TC_TF32X3"
OPS = ["NN", "NT", "TN", "TT"]


def _stored(rng, op, rows, cols):
    r, c = si.stored_shape(op, rows, cols)
    return dyadic(rng, r, c)


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 32), (1, 1, 1), (7, 5, 3), (129, 130, 70), (300, 260, 1000),
                                   (256, 384, 96), (1000, 1300, 700)])
def test_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M * 7 + N + K)
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
        got = gpu_sgemm(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N, variant=V)
        ref = oracle.sgemm(ta, tb, A, B, C, alpha, beta)
        check_exact(got, ref, f"tf32x3 {ops} {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("split", [2, 5, 31])
def test_forced_split_k_exact(ops, split):
    ta, tb = ops
    rng = np.random.default_rng(split)
    M, N, K = 150, 260, 1000
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    got = gpu_sgemm(ta, tb, M, N, K, -2.0, A, A.shape[1], B, B.shape[1], 0.5, C, N, variant=V, split=split)
    ref = oracle.sgemm(ta, tb, A, B, C, -2.0, 0.5)
    check_exact(got, ref, f"tf32x3 split={split} {ops}")


@pytest.mark.parametrize("name", [c.name for c in si.CASES])
def test_config_parity(name):
    c = si.case(name)
    d = si.make_case(c)
    out = gpu_sgemm(c.transA, c.transB, c.M, c.N, c.K, c.alpha, d["A"], d["lda"], d["B"], d["ldb"], c.beta,
                    d["C"], d["ldc"], variant=V)
    if c.pad:
        assert np.all(np.isnan(out[:, c.N:]))
    got = out[:, :c.N]
    rows = None if c.M * c.N * c.K <= 1.2e9 else sample_rows(c.M, 24, seed=c.seed)
    ref, S = oracle_rows(c, d, rows)
    g = got if rows is None else got[rows]
    if c.dist == "int":
        check_exact(g, ref, name)
    else:
        worst, frob = check_bound(g, ref, S, c.K, name)
        print(f"{name}: worst err/bound {worst:.3g}, relative Frobenius {frob:.3g}")


@pytest.mark.parametrize("variant", [V, "TMA_128x128"])
@pytest.mark.parametrize("e", [-24, 24])
def test_power_of_two_scaling_is_exact(variant, e):
    """Scaling A and B by 2^e scales every split part, product and sum exactly, so C(2^e A, 2^e B)
    equals 2^(2e) C(A, B) bit for bit (no flushed partial products, no overflow in the split)."""
    rng = np.random.default_rng(50 + e)
    M, N, K = 192, 320, 700
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = np.zeros((M, N), np.float32)
    base = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=variant)
    s = np.float32(2.0 ** e)
    scaled = gpu_sgemm("N", "N", M, N, K, 1.0, A * s, K, B * s, N, 0.0, C, N, variant=variant)
    check_exact(scaled, base * np.float32(2.0 ** (2 * e)), f"{variant} scale 2^{e}")
