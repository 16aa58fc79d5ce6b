"""GPU parity of the small-product kernel (M, N <= 64 in a strided batch: a
persistent SIMT kernel with a 64x64 tile per product, IEEE FP32 FFMA; chosen
by override) against the oracle, through the C ABI.

Values meet the per-element bound (K+2) u S; small dyadic inputs, whose every
partial sum is exact in float32, must match bit for bit.  Padding and gaps hold
NaN, so a read of them poisons a product and a write to them shows.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, gpu_sgemm, to_dev, torch_cuda
from test_batched import OPS, check_batched, gpu_batched, oracle_batched, plan_of, product_view

pytestmark = pytest.mark.gpu


def small_plan(ta, tb, M, N, K, d, batch):
    sg.sgemm_set_variant_override("SMALL", 0)
    try:
        return plan_of(ta, tb, M, N, K, d, batch)["variant_name"]
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


def _dyadic_stack(d, rng, bits=6):
    for name in "ABC":
        X = d["stacks"][name]
        Y = (rng.integers(-(1 << bits), 1 << bits, size=X.shape) / (1 << bits)).astype(np.float32)
        d["stacks"][name] = Y
        d[name] = si.embed_batched(Y, d["ld" + name.lower()], d["stride" + name])
    return d


@pytest.mark.parametrize("shared", ["", "A", "B"])
@pytest.mark.parametrize("ops", OPS)
def test_small_parity(ops, shared):
    """320 ragged products of 36x20x100 (4 K chunks, the last one ragged), padded rows, gaps."""
    ta, tb = ops
    batch, M, N, K = 320, 36, 20, 100
    d = si.make_batched(batch, M, N, K, ta, tb, seed=51, pad=4, gap=4, align=4, shared=shared)
    assert small_plan(ta, tb, M, N, K, d, batch) == "SMALL"
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch, variant="SMALL")
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"small {ops} shared={shared!r}")


@pytest.mark.parametrize("ops", OPS)
def test_small_persistent_rounds(ops):
    """1111 products on the persistent grid (1-2 products per CTA, 4 K chunks each, the last ragged)."""
    ta, tb = ops
    batch, M, N, K = 1111, 52, 44, 124
    d = si.make_batched(batch, M, N, K, ta, tb, seed=58, pad=4, gap=4, align=4)
    sg.sgemm_set_variant_override("SMALL", 0)
    try:
        p = plan_of(ta, tb, M, N, K, d, batch)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert p["variant_name"] == "SMALL" and p["grid_x"] < batch
    got = gpu_batched(ta, tb, M, N, K, 0.5, 1.5, d, batch, variant="SMALL")
    ref, S = oracle_batched(ta, tb, M, N, K, 0.5, 1.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"persistent {ops}")


@pytest.mark.parametrize("ops", OPS)
def test_small_dyadic_exact(ops):
    """Full 64x64 tiles at K = 1024 (32 chunks, kernel forced): bit-exact on dyadic inputs."""
    ta, tb = ops
    batch, M, N, K = 152, 64, 64, 1024
    d = _dyadic_stack(si.make_batched(batch, M, N, K, ta, tb, seed=0, pad=0, gap=8, align=4),
                      np.random.default_rng(52))
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch, variant="SMALL")
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"dyadic {ops}", exact=True)


# (M, N, K): one row or four columns, K below one float4 chunk boundary, exactly one chunk,
# one chunk plus a float4, outputs of one column group, long K forced
EDGE = [(1, 4, 4), (4, 4, 4), (64, 64, 4), (64, 64, 64), (64, 64, 68), (4, 64, 1024), (64, 4, 1024),
        (13, 28, 12), (64, 64, 3000)]


@pytest.mark.parametrize("M,N,K", EDGE, ids=[f"{m}x{n}x{k}" for m, n, k in EDGE])
@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_small_edges_forced(M, N, K, ops):
    """Edge shapes on a short batch."""
    ta, tb = ops
    if ta == "T" and M % 4:
        M = 4 * ((M + 3) // 4)
    batch = 3
    d = si.make_batched(batch, M, N, K, ta, tb, seed=53 + M + N + K, pad=4, gap=4, align=4)
    assert small_plan(ta, tb, M, N, K, d, batch) == "SMALL"
    got = gpu_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch, variant="SMALL")
    ref, S = oracle_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"edge {ops} {M}x{N}x{K}")


def test_small_beta_zero_does_not_read_c():
    """beta = 0: C may hold NaN on entry and the result is alpha op(A) op(B) all the same."""
    batch, M, N, K = 400, 64, 48, 64
    d = si.make_batched(batch, M, N, K, "N", "T", seed=54, pad=0, gap=0, align=4)
    assert small_plan("N", "T", M, N, K, d, batch) == "SMALL"
    d["C"] = np.full_like(d["C"], np.nan)
    got = gpu_batched("N", "T", M, N, K, 0.75, 0.0, d, batch, variant="SMALL")
    zero = dict(d, C=np.zeros_like(d["C"]))
    ref, S = oracle_batched("N", "T", M, N, K, 0.75, 0.0, zero, batch)
    check_batched(got, ref, S, d, batch, M, N, K, "beta=0 over NaN C")


@pytest.mark.parametrize("ops", ["NN", "TN"])
def test_small_scalar_c_path_with_guard_bands(ops):
    """C 4 bytes past 16-byte alignment, ldc % 4 == 1, NaN around every product: scalar stores only."""
    torch = torch_cuda()
    ta, tb = ops
    batch, M, N, K, ldc = 400, 40, 24, 72, 25
    d = si.make_batched(batch, M, N, K, ta, tb, seed=55, pad=4, gap=4, align=4)
    strideC = M * ldc + 3
    C = si.embed_batched(d["stacks"]["C"], ldc, strideC)
    buf = np.concatenate([np.full(1, np.nan, np.float32), C, np.full(ldc, np.nan, np.float32)])
    dbuf = to_dev(buf)
    c_ptr = dbuf.data_ptr() + 4
    sg.sgemm_set_variant_override("SMALL", 0)
    try:
        plan = sg.sgemm_plan_strided_batched(ta, tb, M, N, K, 1.0, 1 << 20, d["lda"], 1 << 20, d["ldb"], 0.5, c_ptr,
                                             ldc, d["strideA"], d["strideB"], strideC, batch)
        assert plan["variant_name"] == "SMALL"
        sg.sgemm_strided_batched(ta, tb, M, N, K, 1.0, to_dev(d["A"]), d["lda"], to_dev(d["B"]), d["ldb"], 0.5,
                                 c_ptr, ldc, d["strideA"], d["strideB"], strideC, batch)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    out = dbuf.cpu().numpy()
    assert np.isnan(out[0]) and np.all(np.isnan(out[1 + C.size:]))
    got = out[1:1 + C.size]
    dc = dict(d, C=C, ldc=ldc, strideC=strideC)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.0, 0.5, dc, batch)
    check_batched(got, ref, S, dc, batch, M, N, K, f"scalar C {ops}")


def test_small_non_finite_follow_ieee():
    """Inf and NaN inputs give the non-finite pattern of IEEE arithmetic (the FFMA path keeps Inf)."""
    batch, M, N, K = 320, 16, 16, 128
    d = si.make_batched(batch, M, N, K, "N", "N", seed=56, pad=0, gap=0, align=4)
    assert small_plan("N", "N", M, N, K, d, batch) == "SMALL"
    A, B = d["stacks"]["A"].copy(), d["stacks"]["B"].copy()
    A[0, 3, 70] = np.inf          # row 3 of product 0: +-Inf where B[70, n] != 0
    A[1, 5, 10] = np.nan          # row 5 of product 1: NaN
    B[2, 100, 7] = -np.inf        # column 7 of product 2: +-Inf
    A[3, 2, 5] = np.inf           # product 3: Inf * 0 = NaN in row 2, column 9
    B[3, 5, :] = 1.0
    B[3, 5, 9] = 0.0
    for name, X in (("A", A), ("B", B)):
        d["stacks"][name] = X
        d[name] = si.embed_batched(X, d["ld" + name.lower()], d["stride" + name])
    got = gpu_batched("N", "N", M, N, K, 1.0, 0.0, d, batch, variant="SMALL")
    ref = oracle.sgemm_strided_batched("N", "N", M, N, K, 1.0, d["A"], d["lda"], d["strideA"], d["B"], d["ldb"],
                                       d["strideB"], 0.0, d["C"], d["ldc"], d["strideC"], batch)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isposinf(got), np.isposinf(ref)) and np.array_equal(np.isneginf(got), np.isneginf(ref))
    assert np.isnan(product_view(got, 3, M, N, d["ldc"], d["strideC"])[2, 9])
    assert np.isposinf(product_view(got, 3, M, N, d["ldc"], d["strideC"])[2, 0])


def test_small_full_workload_every_product():
    """The benchmark's 8192 products of 64x64x64 in the launch it times: every element against the oracle."""
    c = si.batched_case("batched_small_8192x64x64x64")
    d = si.make_batched(c.batch, c.M, c.N, c.K, c.transA, c.transB, seed=c.seed, dist=c.dist, shared=c.shared,
                        c_init="uniform" if c.beta != 0 else "zero")
    assert small_plan(c.transA, c.transB, c.M, c.N, c.K, d, c.batch) == "SMALL"
    got = gpu_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, c.beta, d, c.batch, variant="SMALL")
    ref, S = oracle_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, c.beta, d, c.batch)
    check_batched(got, ref, S, d, c.batch, c.M, c.N, c.K, c.name)


def test_small_single_product_entry_points_agree():
    """One product forced onto the kernel: sgemm() and sgemm_noalloc() give identical bits, within bound."""
    rng = np.random.default_rng(57)
    M, N, K = 60, 52, 300
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = (2 * rng.random((M, N)) - 1).astype(np.float32)
    one = gpu_sgemm("N", "N", M, N, K, 1.25, A, K, B, N, -1.0, C, N, variant="SMALL")
    torch = torch_cuda()
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    sg.sgemm_set_variant_override("SMALL", 0)
    try:
        sg.sgemm_noalloc("N", "N", M, N, K, 1.25, dA, K, dB, N, -1.0, dC, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    check_exact(dC.cpu().numpy(), one, "noalloc vs sgemm")
    ref, S = oracle.sgemm("N", "N", A, B, C, 1.25, -1.0, want_bound=True)
    check_bound(one, ref, S, K, "single product")
