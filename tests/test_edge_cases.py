"""GPU edge cases of the boundary and the kernels: tiny and ragged shapes, every
operand layout, unaligned pointers and leading dimensions, special alpha/beta
and K values, guard bands around C, forced variants and K splits, streams,
determinism, the transpose identity, and the bounded-wait self-test.

Dyadic inputs (multiples of 2^-6) keep every partial sum exact in float32, so
those cases must equal the oracle bit for bit whatever the summation order.
"""
import itertools

import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, to_dev

pytestmark = pytest.mark.gpu

OPS = ["NN", "NT", "TN", "TT"]


def stored(rng, op, rows, cols, pad=0, fill="dyadic"):
    r, c = si.stored_shape(op, rows, cols)
    X = dyadic(rng, r, c) if fill == "dyadic" else si.uniform_pm1(r, c, int(rng.integers(1 << 30)))
    return si.embed_padded(X, c + pad) if pad else X


def ld_of(X):
    return X.shape[1]


def oracle_ref(ta, tb, A, B, C, alpha, beta, M, N, K):
    Al = A[:, :(M if ta == "T" else K)]
    Bl = B[:, :(K if tb == "T" else N)]
    return oracle.sgemm(ta, tb, Al, Bl, C[:, :N], alpha, beta, M=M, N=N, K=K, want_bound=True)


SHAPES = [(1, 1, 1), (2, 3, 5), (7, 5, 3), (17, 13, 31), (33, 65, 16), (64, 64, 32), (65, 127, 33),
          (129, 130, 70), (128, 256, 96), (200, 72, 129), (1, 300, 257), (300, 1, 64), (5, 7, 1000)]


@pytest.mark.parametrize("variant", ["AUTO", "GENERIC", "TMA_128x128", "TMA_64x256"])
@pytest.mark.parametrize("ops", OPS)
def test_small_shapes_exact(variant, ops):
    ta, tb = ops
    rng = np.random.default_rng(hash((variant, ops)) & 0xFFFF)
    for M, N, K in SHAPES:
        A, B = stored(rng, ta, M, K), stored(rng, tb, K, N)
        C = dyadic(rng, M, N)
        for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
            got = gpu_sgemm(ta, tb, M, N, K, alpha, A, ld_of(A), B, ld_of(B), beta, C, N, variant=variant)
            ref, _ = oracle_ref(ta, tb, A, B, C, alpha, beta, M, N, K)
            check_exact(got, ref, f"{variant} {ops} {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("variant,split", [("TMA_128x128", 2), ("TMA_128x128", 7), ("TMA_64x256", 5),
                                           ("GENERIC", 4)])
def test_forced_split_k_exact(ops, variant, split):
    ta, tb = ops
    rng = np.random.default_rng(split)
    M, N, K = 150, 260, 1000
    A, B = stored(rng, ta, M, K), stored(rng, tb, K, N)
    C = dyadic(rng, M, N)
    got = gpu_sgemm(ta, tb, M, N, K, -2.0, A, ld_of(A), B, ld_of(B), 0.5, C, N, variant=variant, split=split)
    ref, _ = oracle_ref(ta, tb, A, B, C, -2.0, 0.5, M, N, K)
    check_exact(got, ref, f"{variant} split={split} {ops}")


@pytest.mark.parametrize("ops", OPS)
def test_unaligned_operands_take_edge_path(ops):
    """Bases off 16-byte alignment and leading dimensions not multiples of 4."""
    ta, tb = ops
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    M, N, K = 203, 157, 301
    A = stored(rng, ta, M, K, pad=3)
    B = stored(rng, tb, K, N, pad=1)
    C = dyadic(rng, M, N + 5)
    plan = sg.sgemm_plan(ta, tb, M, N, K, 1.0, 4, ld_of(A), 4, ld_of(B), 1.0, 4, N + 5, sm_count=152)
    assert plan["variant_name"] == "GENERIC"
    # copy each operand one float past a 16-byte boundary
    dA = torch.zeros(A.size + 1, device="cuda"); dA[1:] = to_dev(A.reshape(-1))
    dB = torch.zeros(B.size + 3, device="cuda"); dB[3:] = to_dev(B.reshape(-1))
    dC = torch.zeros(C.size + 2, device="cuda"); dC[2:] = to_dev(C.reshape(-1))
    sg.sgemm(ta, tb, M, N, K, 1.0, dA.data_ptr() + 4, ld_of(A), dB.data_ptr() + 12, ld_of(B), 1.0,
             dC.data_ptr() + 8, N + 5)
    assert sg.sgemm_sync_status() == 0
    got = dC[2:].cpu().numpy().reshape(M, N + 5)
    ref, _ = oracle_ref(ta, tb, A, B, C, 1.0, 1.0, M, N, K)
    check_exact(got[:, :N], ref, f"unaligned {ops}")
    assert np.array_equal(got[:, N:], C[:, N:]), "columns past N were written"


@pytest.mark.parametrize("variant", ["AUTO", "GENERIC", "TC_TF32X3", "TC_PAIR", "TC_PRESPLIT"])
def test_beta_zero_does_not_read_nan_c(variant):
    rng = np.random.default_rng(3)
    M, N, K = 300, 260, 200
    A, B = dyadic(rng, M, K), dyadic(rng, K, N)
    C = np.full((M, N), np.nan, np.float32)
    got = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=variant)
    ref, _ = oracle_ref("N", "N", A, B, np.zeros_like(C), 1.0, 0.0, M, N, K)
    check_exact(got, ref, "beta=0 with NaN C")


def test_alpha_zero_and_k_zero_scale_c():
    rng = np.random.default_rng(4)
    M, N = 129, 77
    C = dyadic(rng, M, N)
    nanA = np.full((M, 64), np.nan, np.float32)
    nanB = np.full((64, N), np.nan, np.float32)
    for beta in (0.0, -0.5, 2.0):
        got = gpu_sgemm("N", "N", M, N, 64, 0.0, nanA, 64, nanB, N, beta, C, N)   # alpha = 0: A, B unread
        check_exact(got, (np.float64(beta) * C).astype(np.float32), f"alpha=0 beta={beta}")
    torch = pytest.importorskip("torch")
    dC = to_dev(C)
    sg.sgemm("N", "T", M, N, 0, 1.0, None, 1, None, 1, -0.5, dC, N)                 # K = 0
    assert sg.sgemm_sync_status() == 0
    check_exact(dC.cpu().numpy(), (-0.5 * C.astype(np.float64)).astype(np.float32), "K=0")


def test_zero_m_or_n_is_noop():
    torch = pytest.importorskip("torch")
    dC = torch.full((4, 4), 7.0, device="cuda")
    assert sg.sgemm("N", "N", 0, 4, 4, 1.0, dC, 4, dC, 4, 0.0, dC, 4) == 0
    assert sg.sgemm("N", "N", 4, 0, 4, 1.0, dC, 4, dC, 4, 0.0, dC, 4) == 0
    torch.cuda.synchronize()
    assert bool((dC == 7.0).all())


@pytest.mark.parametrize("variant", ["AUTO", "GENERIC", "TMA_64x256", "TC_TF32X3", "TC_PAIR", "TC_PRESPLIT"])
def test_guard_bands_around_c(variant):
    """C lives inside a NaN-filled buffer (rows above/below, columns past N): only C changes."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    M, N, K, ldc = 131, 133, 97, 140
    A, B = dyadic(rng, M, K), dyadic(rng, K, N)
    C = dyadic(rng, M, N)
    buf = np.full((M + 4, ldc), np.nan, np.float32)
    buf[2:2 + M, :N] = C
    dbuf = to_dev(buf)
    sg.sgemm_set_variant_override(variant, 0)
    try:
        sg.sgemm("N", "N", M, N, K, 1.0, to_dev(A), K, to_dev(B), N, 1.0, dbuf.data_ptr() + 2 * ldc * 4, ldc)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    out = dbuf.cpu().numpy()
    ref, _ = oracle_ref("N", "N", A, B, C, 1.0, 1.0, M, N, K)
    check_exact(out[2:2 + M, :N], ref, "guarded C")
    assert np.all(np.isnan(out[:2])) and np.all(np.isnan(out[2 + M:])) and np.all(np.isnan(out[2:2 + M, N:]))


def test_random_inputs_within_bound_all_ops():
    rng = np.random.default_rng(6)
    M, N, K = 513, 385, 1537
    for ta, tb in OPS:
        A = stored(rng, ta, M, K, fill="uniform")
        B = stored(rng, tb, K, N, fill="uniform")
        C = si.uniform_pm1(M, N, 9)
        got = gpu_sgemm(ta, tb, M, N, K, 1.5, A, ld_of(A), B, ld_of(B), -0.5, C, N)
        ref, S = oracle_ref(ta, tb, A, B, C, 1.5, -0.5, M, N, K)
        check_bound(got, ref, S, K, f"random {ta}{tb}")


@pytest.mark.parametrize("variant", ["AUTO", "TMA_128x128", "TC_TF32X3", "TC_PAIR", "TC_PRESPLIT"])
def test_deterministic_and_transpose_identity(variant):
    """Two runs are bit-identical; sgemm('T','T', B, A) is the transpose of sgemm('N','N', A, B).

    The FP32 FFMA kernel sums the same products in the same order for both, so
    the transpose is exact there; the 3xTF32 kernel adds its two cross terms in
    the opposite order for the transposed problem, so there it must agree within
    the per-element bound.
    """
    torch = pytest.importorskip("torch")
    M, N, K = 1024, 768, 2048
    a_np, b_np = si.uniform_pm1(M, K, 11, 1), si.uniform_pm1(K, N, 11, 2)
    A, B = to_dev(a_np), to_dev(b_np)
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, N, device="cuda")
    Ct = torch.empty(N, M, device="cuda")
    sg.sgemm_set_variant_override(variant, 0)
    try:
        sg.sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C1, N)
        sg.sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C2, N)
        sg.sgemm("T", "T", N, M, K, 1.0, B, N, A, K, 0.0, Ct, M)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    assert torch.equal(C1, C2)
    if variant == "TMA_128x128":
        assert torch.equal(Ct.t(), C1)
    else:
        S = (np.abs(a_np).astype(np.float64) @ np.abs(b_np).astype(np.float64))
        err = np.abs(Ct.t().cpu().numpy().astype(np.float64) - C1.cpu().numpy().astype(np.float64))
        assert np.all(err <= 2 * (K + 2) * 2.0 ** -24 * S)


@pytest.mark.parametrize("ops", OPS)
def test_unaligned_operands_on_tensor_cores(ops):
    """Operands TMA cannot load, large enough for the split-operand kernel: its split pass reads
    them as stored (bases off alignment, ld % 4 != 0) and writes aligned arrays; dyadic inputs
    give the oracle's result bit for bit, random ones meet the bounds."""
    ta, tb = ops
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(22)
    M, N, K = 700, 650, 1203
    for fill in ("dyadic", "uniform"):
        A = stored(rng, ta, M, K, pad=3, fill=fill)
        B = stored(rng, tb, K, N, pad=1, fill=fill)
        C = dyadic(rng, M, N + 5)
        plan = sg.sgemm_plan(ta, tb, M, N, K, 1.0, 4, ld_of(A), 4, ld_of(B), 1.0, 4, N + 5, sm_count=152)
        assert plan["variant_name"] == "TC_PRESPLIT"
        dA = torch.zeros(A.size + 1, device="cuda"); dA[1:] = to_dev(A.reshape(-1))
        dB = torch.zeros(B.size + 3, device="cuda"); dB[3:] = to_dev(B.reshape(-1))
        dC = torch.zeros(C.size + 2, device="cuda"); dC[2:] = to_dev(C.reshape(-1))
        sg.sgemm(ta, tb, M, N, K, 1.0, dA.data_ptr() + 4, ld_of(A), dB.data_ptr() + 12, ld_of(B), 1.0,
                 dC.data_ptr() + 8, N + 5)
        assert sg.sgemm_sync_status() == 0
        got = dC[2:].cpu().numpy().reshape(M, N + 5)
        ref, S = oracle_ref(ta, tb, A, B, C, 1.0, 1.0, M, N, K)
        if fill == "dyadic":
            check_exact(got[:, :N], ref, f"unaligned tensor-core {ops}")
        else:
            check_bound(got[:, :N], ref, S, K, f"unaligned tensor-core {ops}")
        assert np.array_equal(got[:, N:], C[:, N:]), "columns past N were written"


def test_non_default_stream_and_matmul_helper():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    A, B = dyadic(rng, 257, 190), dyadic(rng, 190, 301)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA, dB = to_dev(A), to_dev(B)
        out = sg.matmul(dA, dB, stream=s)
    s.synchronize()
    ref, _ = oracle_ref("N", "N", A, B, np.zeros((257, 301), np.float32), 1.0, 0.0, 257, 301, 190)
    check_exact(out.cpu().numpy(), ref, "stream")
    # op characters 'C'/'c' mean transpose for real data
    outc = sg.matmul(to_dev(np.ascontiguousarray(A.T)), dB, transA="c")
    torch.cuda.synchronize()
    check_exact(outc.cpu().numpy(), ref, "transA='c'")


def test_bounded_wait_selftest_reports_timeout():
    """A kernel whose mbarrier never completes gives up after the limit and reports it."""
    assert sg.sgemm_selftest_wait_timeout(20000) == sg.STATUS["ERR_TIMEOUT"]
    assert sg.sgemm_sync_status() == 0   # the fault word was cleared and the context still works
    test_zero_m_or_n_is_noop()
