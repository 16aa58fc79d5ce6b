"""GPU parity of the 3xTF32 tensor-core kernel (variant TC_TF32X3, op = NN).

Dyadic inputs (multiples of 2^-6) split exactly (lo = 0) and all partial sums
are exact, so those results must equal the oracle bit for bit: this checks
the operand layouts, swizzles, descriptors and the epilogue.  Random inputs
must meet the same per-element and Frobenius bounds as every other path.
"""
import numpy as np
import pytest

import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

V = "TC_TF32X3"


@pytest.mark.parametrize("M,N,K", [(128, 128, 32), (1, 1, 1), (7, 5, 3), (129, 130, 70), (300, 260, 1000),
                                   (256, 384, 96), (1000, 1300, 700)])
def test_dyadic_exact(M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    A, B, C = dyadic(rng, M, K), dyadic(rng, K, N), dyadic(rng, M, N)
    for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
        got = gpu_sgemm("N", "N", M, N, K, alpha, A, K, B, N, beta, C, N, variant=V)
        import oracle
        ref = oracle.sgemm("N", "N", A, B, C, alpha, beta)
        check_exact(got, ref, f"tf32x3 {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("name", ["pr1_random", "pr1_int", "square1024", "square4096", "t2048_NN",
                                  "ragged_NN", "fc_8192x4096x1024", "fc_16384x1024x4096"])
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
