"""GPU parity of sgemm_strided_batched() against the oracle's strided batch.

Every buffer is compared whole: values of each product within the per-element
bound (K+2) u S and the relative Frobenius limit, and the NaN padding and NaN
gaps between matrices unchanged (a kernel that reads them poisons a product,
one that writes them shows there).  Dyadic inputs must match bit for bit on
the tensor-core path.  Everything runs through the C ABI.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, gpu_sgemm, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

OPS = ["NN", "NT", "TN", "TT"]


def gpu_batched(ta, tb, M, N, K, alpha, beta, d, batch, variant=None, split=0):
    torch = torch_cuda()
    dA, dB, dC = to_dev(d["A"]), to_dev(d["B"]), to_dev(d["C"])
    if variant is not None or split:
        sg.sgemm_set_variant_override(variant or "AUTO", split)
    try:
        sg.sgemm_strided_batched(ta, tb, M, N, K, alpha, dA, d["lda"], dB, d["ldb"], beta, dC, d["ldc"],
                                 d["strideA"], d["strideB"], d["strideC"], batch)
    finally:
        if variant is not None or split:
            sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def oracle_batched(ta, tb, M, N, K, alpha, beta, d, batch):
    return oracle.sgemm_strided_batched(ta, tb, M, N, K, alpha, d["A"], d["lda"], d["strideA"], d["B"], d["ldb"],
                                        d["strideB"], beta, d["C"], d["ldc"], d["strideC"], batch, want_bound=True)


def product_view(flat, b, M, N, ldc, strideC):
    return flat[b * strideC:b * strideC + M * ldc].reshape(M, ldc)[:, :N]


def check_batched(got, ref, S, d, batch, M, N, K, what, exact=False):
    assert got.shape == ref.shape
    assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: padding or gap changed (or NaN produced)"
    for b in range(batch):
        g = product_view(got, b, M, N, d["ldc"], d["strideC"])
        r = product_view(ref, b, M, N, d["ldc"], d["strideC"])
        if exact:
            check_exact(g, r, f"{what} product {b}")
        else:
            check_bound(g, r, S[b], K, f"{what} product {b}")


def plan_of(ta, tb, M, N, K, d, batch, alpha=1.0):
    return sg.sgemm_plan_strided_batched(ta, tb, M, N, K, alpha, 1 << 20, d["lda"], 1 << 20, d["ldb"], 0.0,
                                         1 << 20, d["ldc"], d["strideA"], d["strideB"], d["strideC"], batch)


@pytest.mark.parametrize("shared", ["", "A", "B"])
@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("variant,expect", [(None, "TC_TF32X3"), ("TMA_128x128", "TMA_128x128"),
                                            ("TMA_64x256", "TMA_64x256"), ("GENERIC", "GENERIC")])
def test_batched_parity(variant, expect, ops, shared):
    """3 ragged products spanning several tiles, padded rows, gaps between matrices."""
    ta, tb = ops
    batch, M, N, K = 3, 200, 260, 300
    d = si.make_batched(batch, M, N, K, ta, tb, seed=31, pad=4, gap=5, align=4, shared=shared)
    try:
        if variant:
            sg.sgemm_set_variant_override(variant, 0)
        assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == expect
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch, variant=variant)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"{expect} {ops} shared={shared!r}")


def _dyadic_batched(rng, batch, M, N, K, ta, tb, shared=""):
    d = si.make_batched(batch, M, N, K, ta, tb, seed=0, pad=4, gap=8, align=4, shared=shared)
    for name in "ABC":
        X = d["stacks"][name]
        Y = (rng.integers(-64, 64, size=X.shape) / 64).astype(np.float32)
        d["stacks"][name] = Y
        d[name] = si.embed_batched(Y, d["ld" + name.lower()], d["stride" + name])
    return d


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("shared", ["", "B"])
def test_batched_dyadic_exact(ops, shared):
    """Dyadic inputs split exactly on the tensor cores: bit-exact against the oracle."""
    ta, tb = ops
    rng = np.random.default_rng(41)
    batch, M, N, K = 5, 130, 200, 96
    d = _dyadic_batched(rng, batch, M, N, K, ta, tb, shared)
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"dyadic {ops}", exact=True)


@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_batched_odd_strides_on_tensor_cores(ops):
    """Strides and leading dimensions that are not multiples of 4 floats on a batch large enough for
    the split-operand kernel (its split pass reads any layout), a shared B among them."""
    ta, tb = ops
    batch, M, N, K = 6, 300, 270, 601
    d = si.make_batched(batch, M, N, K, ta, tb, seed=33, pad=1, gap=3, align=1, shared="B")
    assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == "TC_PRESPLIT"
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"odd strides tensor cores {ops}")


@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_batched_odd_strides_take_generic(ops):
    """Strides that are not multiples of 4 floats: the any-alignment kernel, same bounds."""
    ta, tb = ops
    batch, M, N, K = 4, 97, 70, 131
    d = si.make_batched(batch, M, N, K, ta, tb, seed=32, pad=1, gap=3, align=1)
    assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == "GENERIC"
    got = gpu_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch)
    ref, S = oracle_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"odd strides {ops}")


@pytest.mark.parametrize("variant", [None, "TMA_128x128", "GENERIC"])
@pytest.mark.parametrize("split", [0, 3])
def test_batched_split_k(variant, split):
    """Few tiles in all: K split across the whole batch (planner's choice, or forced), then the reduction."""
    batch, M, N, K = 2, 64, 384, 8192
    d = si.make_batched(batch, M, N, K, "N", "T", seed=33, dist="fc", pad=0, gap=4, align=4)
    if split == 0 and variant is None:
        assert plan_of("N", "T", M, N, K, d, batch)["split_k"] > 1
    got = gpu_batched("N", "T", M, N, K, 1.0, 0.5, d, batch, variant=variant, split=split)
    ref, S = oracle_batched("N", "T", M, N, K, 1.0, 0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"split {variant} {split}")


def test_batched_many_small_products():
    """2000 ragged products of 33x17x65: one launch, every product correct."""
    batch, M, N, K = 2000, 33, 17, 65
    d = si.make_batched(batch, M, N, K, "N", "N", seed=34, pad=3, gap=0, align=4)
    got = gpu_batched("N", "N", M, N, K, 1.0, 1.0, d, batch)
    ref, S = oracle_batched("N", "N", M, N, K, 1.0, 1.0, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, "many small")


@pytest.mark.parametrize("ops", OPS)
def test_batched_equals_single_calls(ops):
    """With the K split pinned to 1, product b is bit-identical to sgemm() on that product alone."""
    ta, tb = ops
    batch, M, N, K = 3, 150, 140, 250
    d = si.make_batched(batch, M, N, K, ta, tb, seed=35, pad=4, gap=4, align=4)
    got = gpu_batched(ta, tb, M, N, K, 1.25, -1.0, d, batch, split=1)
    for b in range(batch):
        a_rows = si.stored_shape(ta, M, K)[0]
        b_rows = si.stored_shape(tb, K, N)[0]
        A = d["A"][b * d["strideA"]:b * d["strideA"] + a_rows * d["lda"]].reshape(a_rows, d["lda"])
        B = d["B"][b * d["strideB"]:b * d["strideB"] + b_rows * d["ldb"]].reshape(b_rows, d["ldb"])
        C = d["C"][b * d["strideC"]:b * d["strideC"] + M * d["ldc"]].reshape(M, d["ldc"])
        one = gpu_sgemm(ta, tb, M, N, K, 1.25, A, d["lda"], B, d["ldb"], -1.0, C, d["ldc"], split=1)
        check_exact(product_view(got, b, M, N, d["ldc"], d["strideC"]), one[:, :N], f"{ops} product {b}")


def test_batched_alpha_zero_and_empty():
    """alpha = 0 scales every product's C (gaps untouched); batch_count 0 and M = 0 do nothing."""
    batch, M, N, K = 4, 50, 30, 20
    d = si.make_batched(batch, M, N, K, "N", "N", seed=36, pad=2, gap=6, align=1)
    got = gpu_batched("N", "N", M, N, K, 0.0, -2.0, d, batch)
    ref, S = oracle_batched("N", "N", M, N, K, 0.0, -2.0, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, "alpha=0", exact=True)
    got0 = gpu_batched("N", "N", M, N, K, 0.0, 0.0, d, batch)
    ref0, S0 = oracle_batched("N", "N", M, N, K, 0.0, 0.0, d, batch)
    check_batched(got0, ref0, S0, d, batch, M, N, K, "alpha=0 beta=0", exact=True)
    same = gpu_batched("N", "N", M, N, K, 1.0, 1.0, d, 0)
    assert np.array_equal(same, d["C"], equal_nan=True)
    assert sg.sgemm_strided_batched("N", "N", 0, N, K, 1.0, None, K, None, N, 1.0, None, N, 0, 0, 0, 5) == 0


@pytest.mark.parametrize("name", [c.name for c in si.BATCHED_CASES])
def test_batched_workloads_sampled(name):
    """The benchmark's batched workloads at full size, in the launch the benchmark times:
    sampled products and rows against the oracle."""
    c = si.batched_case(name)
    torch = torch_cuda()
    d = si.make_batched(c.batch, c.M, c.N, c.K, c.transA, c.transB, seed=c.seed, dist=c.dist, shared=c.shared,
                        c_init="uniform" if c.beta != 0 else "zero")
    got = gpu_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, c.beta, d, c.batch)
    rng = np.random.default_rng(c.seed)
    products = sorted({0, c.batch - 1, *rng.choice(c.batch, size=min(4, c.batch), replace=False).tolist()})
    rows = sorted({0, c.M - 1, *rng.choice(c.M, size=min(24, c.M), replace=False).tolist()})
    for b in products:
        A = d["stacks"]["A"][0 if "A" in c.shared else b]
        B = d["stacks"]["B"][0 if "B" in c.shared else b]
        C = d["stacks"]["C"][b]
        Ar = np.ascontiguousarray(A[rows, :] if c.transA == "N" else A[:, rows])
        ref, S = oracle.sgemm(c.transA, c.transB, Ar, B, np.ascontiguousarray(C[rows, :]), c.alpha, c.beta,
                              M=len(rows), N=c.N, K=c.K, want_bound=True)
        g = product_view(got, b, c.M, c.N, d["ldc"], d["strideC"])[rows, :]
        check_bound(g, ref, S, c.K, f"{name} product {b}")
    del torch
