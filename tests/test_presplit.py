"""GPU parity of the split-operand 3xTF32 kernel (variant TC_PRESPLIT).

A split pass writes op(A) and op(B) once per call as K-contiguous TF32 hi
and FP32 lo arrays in the workspace (transposing where the stored rows do
not run along K); the CTA-pair GEMM then computes 256 x 256 tiles with both
operands read by the tensor cores from shared memory.  Shapes cover every
operand layout, edges where the odd CTA's rows or B columns fall outside the
matrix, tiles shared between clusters, strided batches with shared operands,
and the caller-workspace entry point.  Dyadic inputs split exactly, so those
results equal the oracle bit for bit; random inputs meet the per-element and
Frobenius bounds; and with one cluster per tile the sums are formed in the
other tensor-core kernels' order, so the results agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, oracle_rows, sample_rows, torch_cuda
from test_batched import _dyadic_batched, check_batched, gpu_batched, oracle_batched, plan_of

pytestmark = pytest.mark.gpu

V = "TC_PRESPLIT"
OPS = ["NN", "NT", "TN", "TT"]


def _stored(rng, op, rows, cols):
    r, c = si.stored_shape(op, rows, cols)
    return dyadic(rng, r, c)


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 32), (1, 1, 4), (7, 5, 4), (128, 128, 64), (129, 200, 70),
                                   (300, 260, 1000), (512, 384, 96), (1000, 1300, 700), (64, 600, 132)])
def test_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M * 7 + N + K)
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
        got = gpu_sgemm(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N, variant=V)
        ref = oracle.sgemm(ta, tb, A, B, C, alpha, beta)
        check_exact(got, ref, f"presplit {ops} {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("split", [2, 5, 31])
def test_forced_split_k_exact(ops, split):
    """Every tile shared by `split` clusters: partial sums in both CTAs' slots, added by the fixup."""
    ta, tb = ops
    rng = np.random.default_rng(split)
    M, N, K = 300, 520, 1000
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    got = gpu_sgemm(ta, tb, M, N, K, -2.0, A, A.shape[1], B, B.shape[1], 0.5, C, N, variant=V, split=split)
    ref = oracle.sgemm(ta, tb, A, B, C, -2.0, 0.5)
    check_exact(got, ref, f"presplit split={split} {ops}")


def test_plan_shape():
    sg.sgemm_set_variant_override(V, 0)
    try:
        p = sg.sgemm_plan("N", "N", 4096, 4096, 4096, 1.5, 1 << 20, 4096, 1 << 20, 4096, -0.5, 1 << 20, 4096, 152)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    # 16 x 16 tiles of 256 x 256 on 76 clusters: 3 whole rounds, then the last 28 tiles by stream-K
    assert (p["variant_name"], p["tile_m"], p["tile_n"], p["grid_x"], p["threads"]) == (V, 256, 256, 152, 320)
    assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (228, 28, 4)
    # slots (2 per CTA, 128 x 256 floats) + hi and lo of A and B
    assert p["workspace_bytes"] == 2 * 152 * 128 * 256 * 4 + 4 * 4096 * 4096 * 4


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
def test_same_sums_as_other_tensor_core_kernels(M, N, K):
    """One cluster (or CTA) per tile, no stream-K: every element is summed in the same order.
    (A's rows are padded to a multiple of 4 floats, so TMA can load it for the one-CTA kernel.)"""
    rng = np.random.default_rng(K)
    lda = (K + 3) // 4 * 4
    A = si.embed_padded((2 * rng.random((M, K)) - 1).astype(np.float32), lda)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = (2 * rng.random((M, N)) - 1).astype(np.float32)
    for v in ("TC_TF32X3", V):
        sg.sgemm_set_variant_override(v, 1)
        try:
            assert sg.sgemm_plan("N", "N", M, N, K, 1.5, 1 << 20, lda, 1 << 20, N, -0.5, 1 << 20, N)["variant_name"] == v
        finally:
            sg.sgemm_set_variant_override("AUTO", 0)
    one = gpu_sgemm("N", "N", M, N, K, 1.5, A, lda, B, N, -0.5, C, N, variant="TC_TF32X3", split=1)
    pre = gpu_sgemm("N", "N", M, N, K, 1.5, A, lda, B, N, -0.5, C, N, variant=V, split=1)
    check_exact(pre, one, f"presplit vs one-CTA {M}x{N}x{K}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("shared", ["", "A", "B"])
def test_batched_dyadic_exact(ops, shared):
    """Strided batches: ragged products, padded rows, gaps, shared operands (split once)."""
    ta, tb = ops
    rng = np.random.default_rng(44)
    batch, M, N, K = 5, 300, 200, 96
    d = _dyadic_batched(rng, batch, M, N, K, ta, tb, shared)
    sg.sgemm_set_variant_override(V, 0)
    try:
        assert plan_of(ta, tb, M, N, K, d, batch)["variant_name"] == V
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    got = gpu_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch, variant=V)
    ref, S = oracle_batched(ta, tb, M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, f"presplit batched {ops} shared={shared!r}", exact=True)


def test_batched_random_stream_k():
    batch, M, N, K = 3, 200, 260, 3000
    d = si.make_batched(batch, M, N, K, "N", "T", seed=36, pad=4, gap=5, align=4)
    got = gpu_batched("N", "T", M, N, K, 1.5, -0.5, d, batch, variant=V)
    ref, S = oracle_batched("N", "T", M, N, K, 1.5, -0.5, d, batch)
    check_batched(got, ref, S, d, batch, M, N, K, "presplit batched stream-K")


def test_caller_workspace_and_noalloc():
    """sgemm_ex with the split arrays in the caller's workspace matches sgemm bit for bit; sgemm_noalloc
    under this override runs the CTA-pair kernel instead (its static scratch holds no split arrays)."""
    torch = torch_cuda()
    rng = np.random.default_rng(8)
    M, N, K = 1536, 1280, 1024
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = [torch.zeros((M, N), dtype=torch.float32, device="cuda") for _ in range(3)]
    sg.sgemm_set_variant_override(V, 0)
    try:
        need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, outs[0], N)
        assert need >= 4 * M * K * 4
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, outs[0], N)
        sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, outs[1], N, ws, need)
        sg.sgemm_noalloc("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, outs[2], N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    assert torch.equal(outs[0], outs[1])
    ref, S = oracle.sgemm("N", "N", A, B, np.zeros((M, N), np.float32), 1.0, 0.0, want_bound=True)
    for o in (outs[0], outs[2]):
        check_bound(o.cpu().numpy(), ref, S, K, "presplit / noalloc fallback")
