"""GPU parity of the BF16-input GEMM (sgemm_bf16) with the oracle's BF16-input GEMM.

sgemm_bf16 computes alpha * op(bf16(A)) * op(bf16(B)) + beta * C with FP32
accumulation (bf16: round to 7 fraction bits, ties to even), the other
tensor-core input format for FP32-range data of youngju.dev "CUDA architecture
visualized" (テンソルコア).  The oracle rounds A and B the same way and sums in
double, so each element must meet (K + 2) u S with S taken over the rounded
inputs, and the relative Frobenius error must be <= 1e-6 -- against the BF16
oracle; against the FP32 oracle the error is that of the rounding (about 2^-8
per product).  Dyadic inputs whose values are BF16 values, and the pages'
integer fill, give results equal bit for bit.  Covers every operand layout,
ragged and padded shapes, unaligned operands (the rounding pass reads any
alignment), tiles shared by several clusters (fixup, 64-deep K tiles), and
Inf / NaN / near-FLT_MAX inputs.
"""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_bound, check_exact, dyadic, sample_rows, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

OPS = ["NN", "NT", "TN", "TT"]


def gpu_bf16(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, split=0, offset=0):
    """sgemm_bf16 on numpy operands (stored, possibly padded); `offset` floats of misalignment
    in front of A and B."""
    torch = torch_cuda()
    dA = to_dev(np.concatenate([np.zeros(offset, np.float32), A.reshape(-1)]))[offset:]
    dB = to_dev(np.concatenate([np.zeros(offset, np.float32), B.reshape(-1)]))[offset:]
    dC = to_dev(C)
    if split:
        sg.sgemm_set_variant_override("AUTO", split)
    try:
        sg.sgemm_bf16(ta, tb, M, N, K, alpha, dA, lda, dB, ldb, beta, dC, ldc)
    finally:
        if split:
            sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def ref_bf16(c, d, rows=None):
    A = d["A"][:, :(c.M if c.transA == "T" else c.K)]
    B = d["B"][:, :(c.K if c.transB == "T" else c.N)]
    C = d["C"][:, :c.N]
    M = c.M
    if rows is not None:
        A = np.ascontiguousarray(A[:, rows] if c.transA == "T" else A[rows, :])
        C = np.ascontiguousarray(C[rows, :])
        M = len(rows)
    return oracle.sgemm_bf16(c.transA, c.transB, A, B, C, c.alpha, c.beta, M=M, N=c.N, K=c.K, want_bound=True)


CONFIGS = ["pr1_random", "pr1_int", "square1024", "square4096", "t2048_NT", "t2048_TN", "ragged_TT",
           "fc_8192x4096x1024", "skinny_64x4096x16384"]


@pytest.mark.parametrize("name", CONFIGS)
def test_configs_match_bf16_oracle(name):
    c = si.case(name)
    d = si.make_case(c)
    got = gpu_bf16(c.transA, c.transB, c.M, c.N, c.K, c.alpha, d["A"], d["lda"], d["B"], d["ldb"], c.beta,
                   d["C"], d["ldc"])
    if c.pad:
        assert np.all(np.isnan(got[:, c.N:])), "padding columns of C were written"
    got = got[:, :c.N]
    rows = None if c.M * c.N * c.K <= 1.2e9 else sample_rows(c.M, 24, seed=c.seed)
    ref, S = ref_bf16(c, d, rows)
    g = got if rows is None else got[rows]
    if c.dist == "int":
        check_exact(g, ref, name)
    else:
        check_bound(g, ref, S, c.K, f"bf16 {name}")


def test_rounding_is_applied():
    """Against the FP32 oracle the BF16 result is off by about the input rounding (relative
    Frobenius well above 1e-6), against the BF16 oracle it is within the FP32 bounds."""
    c = si.case("square1024")
    d = si.make_case(c)
    got = gpu_bf16("N", "N", c.M, c.N, c.K, 1.0, d["A"], c.K, d["B"], c.N, 0.0, d["C"], c.N)
    fp32 = oracle.sgemm("N", "N", d["A"], d["B"])
    frob32 = np.linalg.norm(got.astype(np.float64) - fp32) / np.linalg.norm(fp32.astype(np.float64))
    assert 1e-4 < frob32 < 2e-2, frob32
    ref, S = oracle.sgemm_bf16("N", "N", d["A"], d["B"], want_bound=True)
    check_bound(got, ref, S, c.K, "bf16 square1024")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 3), (256, 256, 32), (300, 520, 1000), (129, 1000, 77)])
def test_dyadic_exact(ops, M, N, K):
    ta, tb = ops
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = dyadic(rng, *si.stored_shape(ta, M, K))
    B = dyadic(rng, *si.stored_shape(tb, K, N))
    C = dyadic(rng, M, N)
    got = gpu_bf16(ta, tb, M, N, K, 1.5, A, A.shape[1], B, B.shape[1], -0.5, C, N)
    check_exact(got, oracle.sgemm_bf16(ta, tb, A, B, C, 1.5, -0.5), f"bf16 dyadic {ops} {M}x{N}x{K}")


@pytest.mark.parametrize("ops", OPS)
@pytest.mark.parametrize("split", [2, 7])
def test_shared_tiles_fixup(ops, split):
    ta, tb = ops
    M, N, K = 700, 600, 2000
    A = si.uniform_pm1(*si.stored_shape(ta, M, K), 41)
    B = si.uniform_pm1(*si.stored_shape(tb, K, N), 42)
    C = si.uniform_pm1(M, N, 43)
    got = gpu_bf16(ta, tb, M, N, K, -1.0, A, A.shape[1], B, B.shape[1], 2.0, C, N, split=split)
    ref, S = oracle.sgemm_bf16(ta, tb, A, B, C, -1.0, 2.0, want_bound=True)
    check_bound(got, ref, S, K, f"bf16 split={split} {ops}")


@pytest.mark.parametrize("ops", OPS)
def test_unaligned_operands(ops):
    """A and B one float past a 16-byte boundary with leading dimensions that are not multiples
    of 4: the rounding pass reads them element by element."""
    ta, tb = ops
    M, N, K = 333, 277, 501
    ar, ac = si.stored_shape(ta, M, K)
    br, bc = si.stored_shape(tb, K, N)
    A = si.embed_padded(si.uniform_pm1(ar, ac, 44), ac + 3)
    B = si.embed_padded(si.uniform_pm1(br, bc, 45), bc + 1)
    C = si.uniform_pm1(M, N, 46)
    got = gpu_bf16(ta, tb, M, N, K, 1.0, A, A.shape[1], B, B.shape[1], 1.0, C, N, offset=1)
    ref, S = oracle.sgemm_bf16(ta, tb, A[:, :ac], B[:, :bc], C, 1.0, 1.0, M=M, N=N, K=K, want_bound=True)
    check_bound(got, ref, S, K, f"bf16 unaligned {ops}")


def test_special_values():
    """Inf, NaN and values whose BF16 rounding passes the largest BF16 value (which become +-Inf):
    the IEEE results of the rounded inputs, NaN where the oracle has NaN."""
    rng = np.random.default_rng(47)
    M, N, K = 300, 264, 256
    a = dyadic(rng, M, K) + np.float32(2.0)
    b = (np.abs(dyadic(rng, K, N)) + np.float32(0.25)) * np.float32(2.0 ** -20)
    a[3, 5] = np.nan
    a[7, 9] = np.inf
    b[9, 30] = 0.0
    a[11, 2] = -np.inf
    a[20, 4], a[20, 6] = np.inf, -np.inf
    a[40, 1] = np.float32((2 - 2.0 ** -8) * 2.0 ** 127)    # a tie at the top: to even, +Inf
    a[41, 1] = np.float32((2 - 2.0 ** -7) * 2.0 ** 127)    # the largest BF16 value: stays finite
    a[50, 3] = np.array([0x7F800001], np.uint32).view(np.float32)[0]  # NaN, payload in the dropped bits
    c = dyadic(rng, M, N)
    got = gpu_bf16("N", "N", M, N, K, 1.5, a, K, b, N, -0.5, c, N)
    ref = oracle.sgemm_bf16("N", "N", a, b, c, 1.5, -0.5)
    assert np.isposinf(ref[40, 0]) and np.all(np.isfinite(ref[41])) and np.all(np.isnan(ref[50]))
    bad = ~((got == ref) | (np.isnan(got) & np.isnan(ref)))
    finite = np.isfinite(ref) & np.isfinite(got)
    # the finite parts are within the bound (dyadic rows exact; row 41 holds a 2^127-sized term)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    _, S = oracle.sgemm_bf16("N", "N", np.where(np.isfinite(a), a, 0).astype(np.float32), b, c, 1.5, -0.5,
                             want_bound=True)
    assert not (bad & ~finite).any(), np.argwhere(bad & ~finite)[:5]
    assert np.all(err[finite] <= (K + 2) * 2.0 ** -24 * S[finite])


def test_argument_errors_and_empty():
    torch = torch_cuda()
    A = torch.zeros(4, 4, device="cuda")
    assert sg.sgemm_bf16("X", "N", 4, 4, 4, 1.0, A, 4, A, 4, 0.0, A, 4, raise_on_error=False) == -1
    assert sg.sgemm_bf16("N", "N", 4, 4, 4, 1.0, A, 3, A, 4, 0.0, A, 4, raise_on_error=False) == -8
    assert sg.sgemm_bf16("N", "N", 0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4) == 0
    C = torch.full((4, 4), 3.0, device="cuda")
    sg.sgemm_bf16("N", "N", 4, 4, 0, 1.0, None, 1, None, 4, 0.5, C, 4)   # K = 0: C = beta C
    torch.cuda.synchronize()
    assert torch.all(C == 1.5)
