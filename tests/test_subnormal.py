"""GPU parity at the bottom of the FP32 range.

Products and partial sums in the subnormal range (normal inputs near 2^-68):
every kernel keeps them, so dyadic inputs give the oracle's results bit for
bit.  Tiny INPUTS (below 2^-115, subnormals included) are where the 3xTF32
split runs out of range: TF32's smallest step is 2^-136, so such an input
reaches the tensor cores only to within 2^-137, and an element's error may
grow by 2^-137 * sum_k(|b_k| over the k with a tiny a_k, |a_k| over the k with
a tiny b_k) beyond the FP32 bound (the library header states this).  The FP32
FFMA kernels meet the FP32 bound there, and so do the TF32- and BF16-input
GEMMs against their oracles (their contract rounds the inputs first).
"""
import numpy as np
import pytest

import oracle
import sgemm_row_major_gb300 as sg
from gpu_util import U, check_exact, dyadic, gpu_sgemm, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

TINY = 2.0 ** -115   # below this an input's 3xTF32 representation error is at most 2^-137, not 2^-21 |x|
LOST = 2.0 ** -137

SHAPES = [(300, 264, 64), (64, 2100, 64), (520, 700, 1000)]
TC_VARIANTS = ["AUTO", "TC_TF32X3", "TC_PAIR", "TC_PRESPLIT", "TC_SKINNY"]
EXACT_VARIANTS = ["TMA_128x128", "TMA_64x256", "GENERIC"]


def _applies(variant, M, N):
    return variant != "TC_SKINNY" or min(M, N) <= 64


def _entry(entry, M, N, K, A, B, C, alpha=1.0, beta=0.0):
    torch = torch_cuda()
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    getattr(sg, entry)("N", "N", M, N, K, alpha, dA, K, dB, N, beta, dC, N)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    return dC.cpu().numpy()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_subnormal_products_exact(M, N, K):
    """Inputs (dyadic, 6-bit significands) times 2^-68: products are multiples of 2^-148 and all
    partial sums lie in the subnormal range, exactly representable; every path gives them bit for
    bit."""
    rng = np.random.default_rng(M + N + K)
    A = dyadic(rng, M, K) * np.float32(2.0 ** -68)
    B = dyadic(rng, K, N) * np.float32(2.0 ** -68)
    C = dyadic(rng, M, N) * np.float32(2.0 ** -140)
    ref = oracle.sgemm("N", "N", A, B, C, 1.0, 1.0)
    assert np.count_nonzero(ref) > 0.9 * ref.size and np.abs(ref).max() < 2.0 ** -120
    for v in TC_VARIANTS + EXACT_VARIANTS:
        if _applies(v, M, N):
            check_exact(gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 1.0, C, N, variant=v), ref, f"{v} {M}x{N}x{K}")
    for entry in ("sgemm_tf32", "sgemm_bf16"):
        check_exact(_entry(entry, M, N, K, A, B, C, 1.0, 1.0), getattr(oracle, entry)("N", "N", A, B, C, 1.0, 1.0),
                    f"{entry} {M}x{N}x{K}")


def test_subnormal_products_grouped_batch_exact():
    """The block-diagonal tensor-core groups (64 x 64 products) on the same tiny products."""
    torch = torch_cuda()
    rng = np.random.default_rng(9)
    P, M, N, K = 200, 64, 64, 64
    A = (dyadic(rng, P * M, K) * np.float32(2.0 ** -68)).reshape(P, M, K)
    B = (dyadic(rng, P * K, N) * np.float32(2.0 ** -68)).reshape(P, K, N)
    C = np.zeros((P, M, N), np.float32)
    assert sg.sgemm_plan_strided_batched("N", "N", M, N, K, 1.0, 1 << 20, K, 1 << 20, N, 0.0, 1 << 20, N,
                                         M * K, K * N, M * N, P)["variant_name"] == "TC_GROUPED"
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    sg.sgemm_strided_batched("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, M * K, K * N, M * N, P)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    for b in range(P):
        check_exact(got[b], oracle.sgemm("N", "N", A[b], B[b], C[b], 1.0, 0.0), f"grouped product {b}")


def _tiny_operands(rng, M, N, K):
    """A: entries k * 2^-130 (below 2^-115 but on TF32's grid) and, a quarter of them, subnormal
    ones k * 2^-143 (bits below TF32's step 2^-136); B: entries near 1 and, 5% of them, k * 2^-143.  Every product is exact in FP32 and the dot products are small enough that the
    tiny inputs' lost parts exceed the FP32 bound."""
    A = dyadic(rng, M, K) * np.float32(2.0 ** -124)
    sub_a = rng.random((M, K)) < 0.25
    A[sub_a] = dyadic(rng, 1, int(sub_a.sum()))[0] * np.float32(2.0 ** -137)
    B = dyadic(rng, K, N) + np.float32(0.5)
    sub_b = rng.random((K, N)) < 0.05
    B[sub_b] = dyadic(rng, 1, int(sub_b.sum()))[0] * np.float32(2.0 ** -137)
    return A, B


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tiny_inputs(M, N, K):
    """FFMA and generic kernels, and the TF32- and BF16-input GEMMs against their oracles: the FP32
    bound (K + 2) u S.  The 3xTF32 kernels: that bound plus the documented loss of tiny inputs,
    2^-137 per tiny input times the other factor -- and the loss is really there (the results
    differ from the exact ones), so the allowance is not vacuous."""
    rng = np.random.default_rng(3 * M + N + K)
    A, B = _tiny_operands(rng, M, N, K)
    C = np.zeros((M, N), np.float32)
    ref, S = oracle.sgemm("N", "N", A, B, C, 1.0, 0.0, want_bound=True)
    bound = (K + 2) * U * S

    def within(got, r, b, what):
        err = np.abs(got.astype(np.float64) - r.astype(np.float64))
        assert np.all(err <= b), f"{what}: worst err/allowance {float(np.max(err / np.maximum(b, 1e-300))):.3g}"

    for v in EXACT_VARIANTS:
        within(gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=v), ref, bound, f"{v} tiny inputs")
    for entry in ("sgemm_tf32", "sgemm_bf16"):
        r, Sr = getattr(oracle, entry)("N", "N", A, B, C, 1.0, 0.0, want_bound=True)
        within(_entry(entry, M, N, K, A, B, C), r, (K + 2) * U * Sr, f"{entry} tiny inputs")
    a64, b64 = np.abs(A.astype(np.float64)), np.abs(B.astype(np.float64))
    extra = LOST * ((a64 < TINY) @ b64 + a64 @ (b64 < TINY))
    for v in TC_VARIANTS:
        if not _applies(v, M, N):
            continue
        got = gpu_sgemm("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N, variant=v)
        within(got, ref, bound + 2.0 * extra, f"{v} tiny inputs")
        assert np.any(got != ref), f"{v}: no tiny-input loss seen (the test lost its point)"
