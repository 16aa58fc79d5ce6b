"""GPU parity of the short-side 3xTF32 kernel (variant TC_SKINNY).

A product with M <= 64 or N <= 64 runs as (long side) x (short side): the
short operand is split once per call into hi and lo arrays in the workspace,
the long one is split in the kernel, tiles are 128 along the long side and 64
along the short side, and when M is the short side the kernel computes
C^T = op(B)^T op(A)^T and writes C transposed.  The cases cover both short
sides, every operand layout, short sides of 1 and of 64, long sides that end
inside a tile, K tails, tiles shared by stream-K and by forced K splits (the
fixup kernel), a short operand TMA could not load (the split pass reads it as
stored), alpha/beta, the benchmark's skinny config, and Inf/NaN inputs.
Dyadic inputs split exactly, so those results equal the oracle bit for bit;
random inputs meet the per-element and Frobenius bounds.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, gpu_sgemm, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

V = "TC_SKINNY"
OPS = ["NN", "NT", "TN", "TT"]


def _stored(rng, op, rows, cols, pad=None):
    """Dyadic stored operand; rows padded to a multiple of 4 floats (TMA) unless `pad` is given."""
    r, c = si.stored_shape(op, rows, cols)
    x = dyadic(rng, r, c)
    pad = (-c) % 4 if pad is None else pad
    return si.embed_padded(x, c + pad) if pad else x


def _plan(ta, tb, M, N, K, lda, ldb, split=0):
    sg.sgemm_set_variant_override(V, split)
    try:
        return sg.sgemm_plan(ta, tb, M, N, K, 1.0, 1 << 20, lda, 1 << 20, ldb, 0.0, 1 << 20, N, 152)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


SHAPES = [(64, 1000, 700), (1, 300, 96), (33, 129, 1000), (64, 4096, 2048), (17, 5000, 33),
          (1000, 64, 700), (300, 1, 96), (129, 33, 1000), (4096, 64, 2048), (5000, 17, 33), (40, 50, 300)]


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M * 7 + N + K)
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    assert _plan(ta, tb, M, N, K, A.shape[1], B.shape[1])["variant_name"] == V
    for alpha, beta in ((1.0, 0.0), (1.5, -0.5)):
        got = gpu_sgemm(ta, tb, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N, variant=V)
        ref = oracle.sgemm(ta, tb, A, B, C, alpha, beta, M=M, N=N, K=K)
        check_exact(got, ref, f"skinny {ops} {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("split", [2, 7, 40])
@pytest.mark.parametrize("M,N", [(64, 520), (520, 64)])
def test_forced_split_k_exact(ops, split, M, N):
    """Every tile shared by `split` CTAs: partial sums in the slots, added by the fixup kernel."""
    ta, tb = ops
    rng = np.random.default_rng(split + M)
    K = 1000
    A, B, C = _stored(rng, ta, M, K), _stored(rng, tb, K, N), dyadic(rng, M, N)
    p = _plan(ta, tb, M, N, K, A.shape[1], B.shape[1], split)
    assert p["variant_name"] == V and p["split_k"] > 1 and p["kernel_launches"] == 3
    got = gpu_sgemm(ta, tb, M, N, K, -2.0, A, A.shape[1], B, B.shape[1], 0.5, C, N, variant=V, split=split)
    ref = oracle.sgemm(ta, tb, A, B, C, -2.0, 0.5, M=M, N=N, K=K)
    check_exact(got, ref, f"skinny split={split} {ops} {M}x{N}")


@pytest.mark.parametrize("ops", OPS)
def test_unaligned_short_operand(ops):
    """The short operand with a leading dimension that is not a multiple of 4 floats: only the long
    operand needs TMA alignment, the split pass reads the short one as stored."""
    ta, tb = ops
    rng = np.random.default_rng(11)
    M, N, K = 48, 900, 531
    A = _stored(rng, ta, M, K, pad=3)
    B = _stored(rng, tb, K, N)
    C = dyadic(rng, M, N)
    assert _plan(ta, tb, M, N, K, A.shape[1], B.shape[1])["variant_name"] == V
    got = gpu_sgemm(ta, tb, M, N, K, 1.25, A, A.shape[1], B, B.shape[1], -1.0, C, N, variant=V)
    ref = oracle.sgemm(ta, tb, A, B, C, 1.25, -1.0, M=M, N=N, K=K)
    check_exact(got, ref, f"skinny unaligned short {ops}")
    # the long operand unaligned instead: the override falls back to the one-CTA kernel's rules
    cols = si.stored_shape(tb, K, N)[1]
    B2 = _stored(rng, tb, K, N, pad=1 if (cols + 1) % 4 else 2)
    assert B2.shape[1] % 4 != 0
    assert _plan(ta, tb, M, N, K, A.shape[1], B2.shape[1])["variant_name"] != V


@pytest.mark.parametrize("ops", ["NN", "TT"])
@pytest.mark.parametrize("M,N,K", [(64, 4096, 16384), (4096, 64, 4096), (50, 3000, 2500)])
def test_random_within_bound(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M + N + K)
    A = (2 * rng.random(si.stored_shape(ta, M, K)) - 1).astype(np.float32)
    B = (2 * rng.random(si.stored_shape(tb, K, N)) - 1).astype(np.float32)
    C = (2 * rng.random((M, N)) - 1).astype(np.float32)
    got = gpu_sgemm(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 1.0, C, N, variant=V)
    ref, S = oracle.sgemm(ta, tb, A, B, C, 1.0, 1.0, want_bound=True)
    worst, frob = check_bound(got, ref, S, K, f"skinny random {ops} {M}x{N}x{K}")
    print(f"skinny {ops} {M}x{N}x{K}: worst err/bound {worst:.3g}, relative Frobenius {frob:.3g}")


def test_skinny_config_parity():
    """The benchmark's skinny config (64 x 4096 x 16384, beta != 0) under this kernel, all of C."""
    c = si.case("skinny_64x4096x16384")
    d = si.make_case(c)
    got = gpu_sgemm(c.transA, c.transB, c.M, c.N, c.K, c.alpha, d["A"], d["lda"], d["B"], d["ldb"], c.beta,
                    d["C"], d["ldc"], variant=V)[:, :c.N]
    ref, S = oracle_rows(c, d, None)
    worst, frob = check_bound(got, ref, S, c.K, c.name)
    print(f"{c.name} on {V}: worst err/bound {worst:.3g}, relative Frobenius {frob:.3g}")


@pytest.mark.parametrize("M,N", [(64, 300), (300, 64)])
@pytest.mark.parametrize("split", [0, 3])
def test_inf_nan_match_oracle(M, N, split):
    """+-Inf, NaN and values whose TF32 rounding overflows, in both operands: the NaN repair gives
    the oracle's IEEE results (same NaN positions and infinities, finite values bit for bit)."""
    K = 256
    rng = np.random.default_rng(M * 3 + split)
    a, b = dyadic(rng, M, K) + np.float32(2.0), np.abs(dyadic(rng, K, N)) + np.float32(0.25)
    a[3, 5] = np.nan
    a[7, 9] = np.inf
    b[9, 30] = 0.0           # C[7, 30] = Inf * 0 = NaN
    a[11, 2] = -np.inf
    a[20, 4], a[20, 6] = np.inf, -np.inf
    b[40, 50] = np.inf       # column 50 +Inf ...
    a[33, 40] = 0.0          # ... except C[33, 50] = NaN
    big = np.float32((2 - 2.0 ** -12) * 2.0 ** 127)
    a[1, 17] = big           # finite product with small entries of b scaled below
    b[17, :] *= np.float32(2.0 ** -20)
    b[17, 9] = 0.0
    c = dyadic(rng, M, N)
    got = gpu_sgemm("N", "N", M, N, K, 1.5, a, K, b, N, -0.5, c, N, variant=V, split=split)
    ref = oracle.sgemm("N", "N", a, b, c, 1.5, -0.5)
    assert np.isnan(ref[7, 30]) and np.isnan(ref[20, 0]) and np.isnan(ref[33, 50]) and np.isposinf(ref[0, 50])
    bad = ~((got == ref) | (np.isnan(got) & np.isnan(ref)))
    assert not bad.any(), f"{M}x{N} split={split}: {int(bad.sum())} differ, first at {tuple(np.argwhere(bad)[0])}"


def test_caller_workspace_and_noalloc():
    """sgemm_ex with the split arrays in the caller's workspace equals sgemm bit for bit; sgemm_noalloc
    (no split arrays) runs the one-CTA kernel instead, within the bound."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    M, N, K = 64, 2048, 3000
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = [torch.zeros((M, N), dtype=torch.float32, device="cuda") for _ in range(3)]
    sg.sgemm_set_variant_override(V, 0)
    try:
        need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, outs[0], N)
        assert need >= 2 * M * K * 4
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
        check_bound(o.cpu().numpy(), ref, S, K, "skinny / noalloc fallback")
