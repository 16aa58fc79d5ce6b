"""GPU parity of the CTA-pair 3xTF32 kernel (variant TC_PAIR, tcgen05 cta_group::2).

The pair kernel computes 256 x 128 tiles on two CTAs of a cluster: each CTA
holds 128 rows of A and half of the tile's B columns, and one thread of the
even CTA issues the MMAs for both.  Shapes here put the second CTA's rows or
B columns wholly or partly outside the matrix (M <= 128, N <= 64, ragged
edges), share tiles between clusters (forced split, stream-K with the fixup
kernel) and run strided batches.  Dyadic inputs split exactly, so those
results must equal the oracle bit for bit; random inputs must meet the
per-element and Frobenius bounds; and with one cluster per tile the pair
kernel sums in the one-CTA kernel's order, so the two agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, oracle_rows, sample_rows
from test_batched import _dyadic_batched, check_batched, gpu_batched, oracle_batched, plan_of

pytestmark = pytest.mark.gpu

V = "TC_PAIR"
OPS = ["NN", "NT", "TN", "TT"]


def _stored(rng, op, rows, cols):
    r, c = si.stored_shape(op, rows, cols)
    return dyadic(rng, r, c)


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("M,N,K", [(256, 128, 32), (1, 1, 1), (7, 5, 3), (128, 64, 64), (129, 65, 70),
                                   (300, 260, 1000), (512, 384, 96), (1000, 1300, 700), (64, 200, 130)])
def test_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M * 7 + N + K)
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
        got = gpu_sgemm(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N, variant=V)
        ref = oracle.sgemm(ta, tb, A, B, C, alpha, beta)
        check_exact(got, ref, f"pair {ops} {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("split", [2, 5, 31])
def test_forced_split_k_exact(ops, split):
    """Every tile shared by `split` clusters: partial sums in both CTAs' slots, added by the fixup."""
    ta, tb = ops
    rng = np.random.default_rng(split)
    M, N, K = 300, 260, 1000
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    got = gpu_sgemm(ta, tb, M, N, K, -2.0, A, A.shape[1], B, B.shape[1], 0.5, C, N, variant=V, split=split)
    ref = oracle.sgemm(ta, tb, A, B, C, -2.0, 0.5)
    check_exact(got, ref, f"pair split={split} {ops}")


def test_plan_shape():
    sg.sgemm_set_variant_override(V, 0)
    try:
        p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 1.5, 1 << 20, 4096, 1 << 20, 4096, -0.5, 1 << 20, 4096, 152)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    # 16 x 32 pair tiles on 76 clusters: 6 whole rounds (456 tiles), the last 56 tiles by stream-K
    assert (p["variant_name"], p["tile_m"], p["tile_n"], p["grid_x"]) == ("TC_PAIR", 256, 128, 152)
    assert (p["dp_tiles"], p["sk_tiles"], p["sk_iters"]) == (456, 56, 56 * 128)
    assert p["workspace_bytes"] == 2 * 152 * 128 * 128 * 4


SCHEDULES = [
    (256 * 19, 512, 64, 0, "whole rounds"),            # 76 pair tiles: 1 round on 76 clusters
    (256 * 20, 512, 64, 0, "ragged rounds"),           # 80 tiles, short K: ragged whole rounds
    (256 * 39, 512, 2048, 0, "rounds + stream-K"),     # 156 tiles: 1 round + 80 stream-K tiles
    (256, 256, 1216 * 32, 0, "stream-K on every cluster"),  # 2 tiles, 1216 K tiles each
    (300, 260, 700, 0, "split per tile"),              # 6 tiles, short K: 5 clusters per tile
    (256, 128, 8192, 64, "forced 64 per tile"),        # one tile shared by 64 clusters
    (4, 4, 32, 0, "one tile one K tile"),
]


@pytest.mark.parametrize("M,N,K,split,what", SCHEDULES, ids=[s[4] for s in SCHEDULES])
def test_schedule_branches_exact(M, N, K, split, what):
    """Every branch of the persistent schedule with clusters as the unit, on small integers (exact)."""
    sg.sgemm_set_variant_override(V, split)
    try:
        p = sg.sgemm_plan("N", "N", M, N, K, 1.0, 1 << 20, K, 1 << 20, N, 0.5, 1 << 20, N, 152)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert p["variant_name"] == V
    if what == "whole rounds":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (76, 0, 1)
    elif what == "ragged rounds":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (80, 0, 1)
    elif what == "rounds + stream-K":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (76, 80, 2)
    elif what == "stream-K on every cluster":
        assert (p["grid_x"], p["dp_tiles"], p["sk_tiles"]) == (152, 0, 2) and p["split_k"] >= 38
    elif what == "split per tile":
        assert (p["grid_x"], p["sk_tiles"]) == (2 * 6 * 5, 6)
    elif what == "forced 64 per tile":
        assert p["grid_x"] == 128 and p["split_k"] == 64
    else:
        assert (p["grid_x"], p["kernel_launches"], p["workspace_bytes"]) == (2, 1, 0)
    rng = np.random.default_rng(M + N + K)
    A, B, C = (rng.integers(-2, 3, size=s).astype(np.float32) for s in ((M, K), (K, N), (M, N)))
    got = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.5, C, N, variant=V, split=split)
    check_exact(got, oracle.sgemm("N", "N", A, B, C, 1.0, 0.5), what)


@pytest.mark.parametrize("name", [c.name for c in si.CASES])
def test_config_parity(name):
    c = si.case(name)
    d = si.make_case(c)
    out = gpu_sgemm(c.transA, c.transB, c.M, c.N, c.K, c.alpha, d["A"], d["lda"], d["B"], d["ldb"], c.beta,
                    d["C"], d["ldc"], variant=V)
    if c.pad:
        assert np.all(np.isnan(out[:, c.N:]))
    got = out[:, :c.N]
    rows = None if c.M * c.N * c.K <= 1.2e9 else sample_rows(c.M, 24, seed=c.seed, tile=256)
    ref, S = oracle_rows(c, d, rows)
    g = got if rows is None else got[rows]
    if c.dist == "int":
        check_exact(g, ref, name)
    else:
        worst, frob = check_bound(g, ref, S, c.K, name)
        print(f"{name}: worst err/bound {worst:.3g}, relative Frobenius {frob:.3g}")


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (777, 1000, 2053)])
def test_same_sums_as_one_cta_kernel(M, N, K):
    """One cluster (or CTA) per tile, no stream-K: every element is summed in the same order."""
    rng = np.random.default_rng(K)
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = (2 * rng.random((M, N)) - 1).astype(np.float32)
    one = gpu_sgemm("N", "N", M, N, K, 1.5, A, K, B, N, -0.5, C, N, variant="TC_TF32X3", split=1)
    pair = gpu_sgemm("N", "N", M, N, K, 1.5, A, K, B, N, -0.5, C, N, variant=V, split=1)
    check_exact(pair, one, f"pair vs one-CTA {M}x{N}x{K}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("shared", ["", "A", "B"])
def test_batched_dyadic_exact(ops, shared):
    """Strided batches on the pair kernel: ragged products, padded rows, gaps, shared operands."""
    ta, tb = ops
    rng = np.random.default_rng(43)
    batch, M, N, K = 5, 300, 200, 96
    d = _dyadic_batched(rng, batch, M, N, K, ta, tb, shared)
    sg.sgemm_set_variant_override(V, 0)
    try:
        assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == V
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch, variant=V)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"pair batched {ops} shared={shared!r}", exact=True)


def test_batched_random_stream_k():
    """Random inputs, a batch whose tiles do not fill the clusters: stream-K across products."""
    batch, M, N, K = 3, 200, 260, 3000
    d = si.make_batched(batch, M, N, K, "N", "T", seed=35, pad=4, gap=5, align=4)
    got = gpu_batched("N", "T", M, N, K, 1.5, -0.5, d, batch, variant=V)
    ref, S = oracle_batched("N", "T", M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, "pair batched stream-K")


def test_noalloc_matches_sgemm():
    """sgemm_noalloc on the pair kernel (stream-K slots in the static scratch) matches sgemm."""
    torch = __import__("torch")
    rng = np.random.default_rng(5)
    M, N, K = 2048, 2048, 2048
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    c2 = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    sg.sgemm_set_variant_override(V, 0)
    try:
        assert sg.sgemm_plan("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, c1, N)["split_k"] > 1
        sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, c1, N)
        sg.sgemm_noalloc("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, c2, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    assert torch.equal(c1, c2)
