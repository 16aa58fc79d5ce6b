"""GPU tests of sgemm_host: the SGEMM entry point for operands in host memory.

Results must equal the oracle bit for bit on dyadic inputs (all partial sums
exact) and meet the error bounds on random inputs, for every operand layout,
padded leading dimensions, beta = 0 with NaN in C, alpha = 0 and K = 0, and
problems whose M is not a multiple of the internal row block.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic

pytestmark = pytest.mark.gpu


def _pinned(x):
    import torch
    t = torch.empty(x.shape, dtype=torch.float32, pin_memory=True)
    t.numpy()[...] = x
    return t


def _run_host(ta, tb, M, N, K, alpha, A, B, C, beta, pinned=True):
    import torch
    hA, hB, hC = (_pinned(x) if pinned else np.ascontiguousarray(x) for x in (A, B, C))
    sg.sgemm_host(ta, tb, M, N, K, alpha, hA, A.shape[1], hB, B.shape[1], beta, hC, C.shape[1])
    torch.cuda.synchronize()
    assert sg.sgemm_sync_status() == 0
    return hC.numpy() if pinned else hC


@pytest.mark.parametrize("ops", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (37, 53, 29), (700, 300, 257), (2100, 517, 300)])
def test_host_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M + N + K)
    A = dyadic(rng, *si.stored_shape(ta, M, K))
    B = dyadic(rng, *si.stored_shape(tb, K, N))
    C = dyadic(rng, M, N)
    for alpha, beta in ((1.0, 0.0), (-1.5, 0.5)):
        got = _run_host(ta, tb, M, N, K, alpha, A, B, C.copy(), beta)
        check_exact(got, oracle.sgemm(ta, tb, A, B, C, alpha, beta), f"host {ops} {M}x{N}x{K}")


def test_host_padded_random_and_pageable():
    c = si.Case("host_ragged", 1537, 901, 777, "T", "N", 1.0, 1.0, 5, "uniform", 3, "uniform")
    d = si.make_case(c)
    for pinned in (True, False):
        got = _run_host("T", "N", c.M, c.N, c.K, 1.0, d["A"], d["B"], d["C"].copy(), 1.0, pinned=pinned)
        assert np.all(np.isnan(got[:, c.N:])), "padding of C was written"
        ref, S = oracle.sgemm("T", "N", d["A"][:, :c.M], d["B"][:, :c.N], d["C"][:, :c.N], 1.0, 1.0, want_bound=True)
        check_bound(got[:, :c.N], ref, S, c.K, f"host padded pinned={pinned}")


def test_host_special_scalars():
    rng = np.random.default_rng(9)
    M, N, K = 300, 200, 100
    A, B = dyadic(rng, M, K), dyadic(rng, K, N)
    nanC = np.full((M, N), np.nan, np.float32)
    got = _run_host("N", "N", M, N, K, 2.0, A, B, nanC, 0.0)
    check_exact(got, oracle.sgemm("N", "N", A, B, None, 2.0, 0.0), "host beta=0 NaN C")
    C = dyadic(rng, M, N)
    got = _run_host("N", "N", M, N, K, 0.0, np.full_like(A, np.nan), np.full_like(B, np.nan), C.copy(), -0.5)
    check_exact(got, (-0.5 * C.astype(np.float64)).astype(np.float32), "host alpha=0")
    assert sg.sgemm_host("N", "N", 0, N, K, 1.0, None, K, None, N, 0.0, None, N) == 0
    assert sg.sgemm_host("X", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, raise_on_error=False) == -1
