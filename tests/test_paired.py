"""GPU parity of the block-diagonal tensor-core mode (products with M, N <= 64
two to a 128x128 tile, with M, N <= 32 four to a tile) against the oracle,
through the C ABI.

Values meet the per-element bound (K+2) u S; dyadic inputs, which the 3xTF32
split represents exactly, must match bit for bit.  Padding and gaps hold NaN,
so a read of them poisons a product and a write to them shows; an odd batch
leaves the last tile's second product missing (zeros read, nothing written).
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, gpu_sgemm, to_dev, torch_cuda
from test_batched import OPS, check_batched, gpu_batched, oracle_batched, plan_of
from test_small import _dyadic_stack

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,group", [(36, 20, 2), (20, 28, 4)], ids=["pairs", "quads"])
@pytest.mark.parametrize("shared", ["", "A", "B"])
@pytest.mark.parametrize("ops", OPS)
def test_paired_parity(ops, shared, M, N, group):
    """305 ragged products of K = 300 (a batch that leaves the last tile short, ragged last K
    tile), padded rows, gaps."""
    ta, tb = ops
    batch, K = 305, 300
    d = si.make_batched(batch, M, N, K, ta, tb, seed=71, pad=4, gap=4, align=4, shared=shared)
    p = plan_of(ta, tb, M, N, K, d, batch)
    assert p["variant_name"] == "TC_GROUPED" and p["tile_m"] == 128 // group
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"paired {ops} shared={shared!r}")


@pytest.mark.parametrize("ops", OPS)
def test_paired_dyadic_exact(ops):
    """Full 64x64 products, K = 512: bit-exact on dyadic inputs."""
    ta, tb = ops
    batch, M, N, K = 311, 64, 64, 512
    d = _dyadic_stack(si.make_batched(batch, M, N, K, ta, tb, seed=0, pad=0, gap=8, align=4),
                      np.random.default_rng(72))
    assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == "TC_GROUPED"
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"paired dyadic {ops}", exact=True)


# (batch, M, N, K): one product, one pair, an odd batch; one row, four columns, K of one float4;
# quads (M, N <= 32) with 1, 2 and 3 products in the last tile
EDGE = [(1, 64, 64, 96), (2, 1, 4, 4), (3, 13, 64, 32), (3, 64, 4, 100), (5, 40, 28, 2000),
        (1, 32, 32, 64), (6, 1, 4, 4), (7, 32, 8, 500), (9, 17, 32, 36)]


@pytest.mark.parametrize("batch,M,N,K", EDGE, ids=[f"{b}x{m}x{n}x{k}" for b, m, n, k in EDGE])
@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_paired_edges_forced(batch, M, N, K, ops):
    """Edge shapes on short batches, with the mode forced (the default needs a pair per SM)."""
    ta, tb = ops
    if ta == "T" and M % 4:
        M = 4 * ((M + 3) // 4)
    d = si.make_batched(batch, M, N, K, ta, tb, seed=73 + M + N + K, pad=4, gap=4, align=4)
    sg.sgemm_set_variant_override("TC_GROUPED", 0)
    try:
        assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == "TC_GROUPED"
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    got = gpu_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch, variant="TC_GROUPED")
    ref, S = oracle_batched(ta, tb, M, N, K, -1.0, 2.0, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"paired edge {ops} {batch}x{M}x{N}x{K}")


def test_paired_beta_zero_does_not_read_c():
    """beta = 0: C may hold NaN on entry and the result is alpha op(A) op(B) all the same."""
    batch, M, N, K = 400, 64, 48, 256
    d = si.make_batched(batch, M, N, K, "N", "T", seed=74, pad=0, gap=0, align=4)
    assert plan_of("N", "T", M, N, K, d, batch)["variant_name"] == "TC_GROUPED"
    d["C"] = np.full_like(d["C"], np.nan)
    got = gpu_batched("N", "T", M, N, K, 0.75, 0.0, d, batch)
    ref, S = oracle_batched("N", "T", M, N, K, 0.75, 0.0, dict(d, C=np.zeros_like(d["C"])), batch)
    check_batched(got, ref, S, d, batch, M, N, K, "paired beta=0 over NaN C")


@pytest.mark.parametrize("ops", ["NN", "TN"])
def test_paired_scalar_c_path_with_guard_bands(ops):
    """C 4 bytes past 16-byte alignment, ldc % 4 == 1, NaN around every product: scalar stores only."""
    torch = torch_cuda()
    ta, tb = ops
    batch, M, N, K, ldc = 401, 40, 24, 200, 25
    d = si.make_batched(batch, M, N, K, ta, tb, seed=75, pad=4, gap=4, align=4)
    strideC = M * ldc + 3
    C = si.embed_batched(d["stacks"]["C"], ldc, strideC)
    buf = np.concatenate([np.full(1, np.nan, np.float32), C, np.full(ldc, np.nan, np.float32)])
    dbuf = to_dev(buf)
    c_ptr = dbuf.data_ptr() + 4
    plan = sg.sgemm_plan_strided_batched(ta, tb, M, N, K, 1.0, 1 << 20, d["lda"], 1 << 20, d["ldb"], 0.5, c_ptr,
                                         ldc, d["strideA"], d["strideB"], strideC, batch)
    assert plan["variant_name"] == "TC_GROUPED"
    sg.sgemm_strided_batched(ta, tb, M, N, K, 1.0, to_dev(d["A"]), d["lda"], to_dev(d["B"]), d["ldb"], 0.5, c_ptr,
                             ldc, d["strideA"], d["strideB"], strideC, batch)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    out = dbuf.cpu().numpy()
    assert np.isnan(out[0]) and np.all(np.isnan(out[1 + C.size:]))
    dc = dict(d, C=C, ldc=ldc, strideC=strideC)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.0, 0.5, dc, batch)
    check_batched(out[1:1 + C.size], ref, S, dc, batch, M, N, K, f"paired scalar C {ops}")


def test_paired_single_product_entry_points_agree():
    """One product forced into the mode: sgemm() and sgemm_noalloc() give identical bits, within bound."""
    rng = np.random.default_rng(76)
    M, N, K = 60, 52, 3000
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = (2 * rng.random((M, N)) - 1).astype(np.float32)
    one = gpu_sgemm("N", "N", M, N, K, 1.25, A, K, B, N, -1.0, C, N, variant="TC_GROUPED")
    torch = torch_cuda()
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    sg.sgemm_set_variant_override("TC_GROUPED", 0)
    try:
        sg.sgemm_noalloc("N", "N", M, N, K, 1.25, dA, K, dB, N, -1.0, dC, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    check_exact(dC.cpu().numpy(), one, "noalloc vs sgemm")
    ref, S = oracle.sgemm("N", "N", A, B, C, 1.25, -1.0, want_bound=True)
    check_bound(one, ref, S, K, "single product")


@pytest.mark.parametrize("name", ["batched_small_8192x64x64x64", "batched_small_k1024_2048x64x64x1024",
                                  "batched_tiny_16384x32x32x32"])
def test_paired_full_workloads_every_product(name):
    """The benchmark's small-product batches in the launch it times: every element against the oracle."""
    c = si.batched_case(name)
    d = si.make_batched(c.batch, c.M, c.N, c.K, c.transA, c.transB, seed=c.seed, dist=c.dist, shared=c.shared,
                        c_init="uniform" if c.beta != 0 else "zero")
    assert plan_of(c.transA, c.transB, c.M, c.N, c.K, d, c.batch)["variant_name"] == "TC_GROUPED"
    got = gpu_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, c.beta, d, c.batch)
    ref, S = oracle_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, c.beta, d, c.batch)
    check_batched(got, ref, S, d, c.batch, c.M, c.N, c.K, c.name)
