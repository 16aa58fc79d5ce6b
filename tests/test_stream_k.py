"""GPU tests of the one-CTA tensor-core kernel's persistent schedule (whole-tile rounds + stream-K).

Every branch of the planner is run on small-integer inputs (-2..2): their
3xTF32 split is exact and every partial sum is an integer below 2^24, so the
results must equal the oracle bit for bit whatever the split of K across CTAs.
The fixup kernel's scalar path (C not 16-byte aligned, ldc % 4 != 0) runs
inside a NaN-filled buffer, so a write outside C or a read of the padding
shows.
"""
import numpy as np
import pytest

import oracle
import sgemm_row_major_gb300 as sg
from gpu_util import check_exact, gpu_sgemm, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


def _ints(rng, rows, cols):
    return rng.integers(-2, 3, size=(rows, cols)).astype(np.float32)


def _case(seed, M, N, K):
    rng = np.random.default_rng(seed)
    return _ints(rng, M, K), _ints(rng, K, N), _ints(rng, M, N)


V = "TC_TF32X3"  # the CTA-pair kernel's schedule is tested in test_pair.py


def _plan(M, N, K, split=0):
    sg.sgemm_set_variant_override(V, split)
    try:
        return sg.sgemm_plan("N", "N", M, N, K, 1.0, 1 << 20, K, 1 << 20, N, 0.5, 1 << 20, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)


# (M, N, K, forced split, what the plan must look like)
SHAPES = [
    (128 * 19, 1024, 64, 0, "whole rounds"),            # 152 tiles: 1 round, no stream-K
    (128 * 20, 1024, 64, 0, "ragged rounds"),           # 160 tiles, short K: ragged whole rounds
    (128 * 39, 1024, 2048, 0, "rounds + stream-K"),     # 312 tiles: 1 round + 160 stream-K tiles
    (128, 256, 2432 * 32, 0, "stream-K on every SM"),   # 2 tiles, 2432 K tiles each
    (300, 260, 700, 0, "split per tile"),               # 9 tiles, short K: 5 CTAs per tile
    (128, 128, 8192, 128, "forced 128 per tile"),       # one tile shared by 128 CTAs
    (4, 4, 32, 0, "one tile one K tile"),
]


@pytest.mark.parametrize("M,N,K,split,what", SHAPES, ids=[s[4] for s in SHAPES])
def test_schedule_branches_exact(M, N, K, split, what):
    p = _plan(M, N, K, split)
    assert p["variant_name"] == "TC_TF32X3"
    if what == "whole rounds":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (152, 0, 1)
    elif what == "ragged rounds":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (160, 0, 1)
    elif what == "rounds + stream-K":
        assert (p["dp_tiles"], p["sk_tiles"], p["kernel_launches"]) == (152, 160, 2)
    elif what == "stream-K on every SM":
        assert (p["grid_x"], p["dp_tiles"], p["sk_tiles"]) == (152, 0, 2) and p["split_k"] >= 76
    elif what == "split per tile":
        assert (p["grid_x"], p["sk_tiles"]) == (45, 9)
    elif what == "forced 128 per tile":
        assert p["grid_x"] == 128 and p["split_k"] == 128
    else:
        assert (p["grid_x"], p["kernel_launches"], p["workspace_bytes"]) == (1, 1, 0)
    A, B, C = _case(M + N + K, M, N, K)
    got = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.5, C, N, variant=V, split=split)
    ref = oracle.sgemm("N", "N", A, B, C, 1.0, 0.5)
    check_exact(got, ref, what)


@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_fixup_scalar_path_with_guard_bands(ops):
    """Stream-K tiles shared by several CTAs, C 4-byte aligned with ldc % 4 == 1."""
    torch = torch_cuda()
    ta, tb = ops
    M, N, K, ldc = 200, 301, 3000, 305
    rng = np.random.default_rng(77)
    A = _ints(rng, *((K, M) if ta == "T" else (M, K)))
    B = _ints(rng, *((N, K) if tb == "T" else (K, N)))
    C = _ints(rng, M, N)
    lda, ldb = A.shape[1], B.shape[1]
    # A and B need 16-byte rows for the tensor-core path: pad them to a multiple of 4 floats
    Ap = np.full((A.shape[0], (lda + 3) // 4 * 4), np.nan, np.float32); Ap[:, :lda] = A
    Bp = np.full((B.shape[0], (ldb + 3) // 4 * 4), np.nan, np.float32); Bp[:, :ldb] = B
    buf = np.full((M + 3, ldc), np.nan, np.float32)
    buf[1:1 + M, :N] = C
    flat = buf.ravel()
    dflat = to_dev(np.concatenate([np.full(1, np.nan, np.float32), flat]))  # C base 4 bytes past 16-byte alignment
    c_ptr = dflat.data_ptr() + 4 + ldc * 4
    plan = sg.sgemm_plan(ta, tb, M, N, K, 1.0, 1 << 20, Ap.shape[1], 1 << 20, Bp.shape[1], 0.5, 1 << 20, ldc)
    assert plan["variant_name"] == "TC_TF32X3" and plan["kernel_launches"] == 2
    sg.sgemm(ta, tb, M, N, K, 1.0, to_dev(Ap), Ap.shape[1], to_dev(Bp), Bp.shape[1], 0.5, c_ptr, ldc)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    out = dflat.cpu().numpy()[1:].reshape(M + 3, ldc)
    ref = oracle.sgemm(ta, tb, A, B, C, 1.0, 0.5)
    check_exact(out[1:1 + M, :N], ref, f"fixup scalar {ops}")
    assert np.all(np.isnan(out[0])) and np.all(np.isnan(out[1 + M:])) and np.all(np.isnan(out[1:1 + M, N:]))


def test_stream_k_is_deterministic():
    """Random inputs, shared tiles: two runs give identical bits (fixed summation order)."""
    rng = np.random.default_rng(3)
    M, N, K = 512, 768, 4096
    A = (2 * rng.random((M, K)) - 1).astype(np.float32)
    B = (2 * rng.random((K, N)) - 1).astype(np.float32)
    C = np.zeros((M, N), np.float32)
    assert _plan(M, N, K)["split_k"] > 1
    for v in (V, "TC_PAIR"):
        one = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=v)
        two = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=v)
        assert np.array_equal(one, two), v
