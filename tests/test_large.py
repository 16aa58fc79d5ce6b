"""GPU tests at sizes whose element offsets pass 2^31: C of one product larger
than 2^31 elements, and strided batches whose product offsets pass it (the
tensor-core kernel, the block-diagonal groups, and the FP32 kernels).  Inputs
are small integers drawn on the device from a seeded generator, so every
result is exact; rows and products on both sides of the 2^31 boundary are
compared with the oracle."""
import numpy as np
import pytest

import oracle
import sgemm_row_major_gb300 as sg
from gpu_util import check_exact, torch_cuda

pytestmark = pytest.mark.gpu

TWO31 = 1 << 31


def _ints(torch, shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(-2, 3, shape, generator=g, device="cuda", dtype=torch.int32).to(torch.float32)


@pytest.mark.parametrize("variant", [None, "TC_PAIR", "TC_TF32X3", "GENERIC", "TMA_128x128"])
def test_c_larger_than_2g_elements(variant):
    torch = torch_cuda()
    M, N, K = 70000, 32772, 32
    assert M * N > TWO31
    dA, dB = _ints(torch, (M, K), 91), _ints(torch, (K, N), 92)
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    if variant:
        sg.sgemm_set_variant_override(variant, 0)
    try:
        sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
    finally:
        if variant:
            sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    boundary = TWO31 // N  # the first row whose offset passes 2^31
    rows = sorted({0, boundary - 1, boundary, boundary + 1, M - 2, M - 1, 12345})
    got = dC[rows].cpu().numpy()
    A = dA[rows].cpu().numpy()
    ref = oracle.sgemm("N", "N", A, dB.cpu().numpy(), np.zeros((len(rows), N), np.float32), 1.0, 0.0)
    check_exact(got, ref, f"rows beyond 2^31 ({variant or 'default'})")
    del dC


@pytest.mark.parametrize("variant,expect", [(None, "TC_PRESPLIT"), ("TC_PAIR", "TC_PAIR"), ("TC_TF32X3", "TC_TF32X3")])
def test_strided_batch_offsets_beyond_2g(variant, expect):
    torch = torch_cuda()
    batch, M, N, K = 3000, 1024, 1024, 32
    assert batch * M * N > TWO31
    dA = _ints(torch, (batch, M, K), 93)
    dB = _ints(torch, (K, N), 94)  # shared by every product (stride 0)
    dC = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
    if variant:
        sg.sgemm_set_variant_override(variant, 0)
    try:
        assert sg.sgemm_plan_strided_batched("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, M * K, 0, M * N,
                                             batch)["variant_name"] == expect
        sg.sgemm_strided_batched("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, M * K, 0, M * N, batch)
    finally:
        if variant:
            sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    first = TWO31 // (M * N)  # the first product whose offset passes 2^31
    B = dB.cpu().numpy()
    for b in sorted({0, first - 1, first, first + 1, batch - 1}):
        ref = oracle.sgemm("N", "N", dA[b].cpu().numpy(), B, np.zeros((M, N), np.float32), 1.0, 0.0)
        check_exact(dC[b].cpu().numpy(), ref, f"product {b}")
    del dC


def test_grouped_batch_offsets_beyond_2g():
    """2.2 million products of 32x32x32, four to a tensor-core tile: operands of 9 GB each."""
    torch = torch_cuda()
    batch, M, N, K = 2_200_000, 32, 32, 32
    assert batch * M * N > TWO31
    dA = _ints(torch, (batch, M, K), 95)
    dB = _ints(torch, (batch, K, N), 96)
    dC = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
    plan = sg.sgemm_plan_strided_batched("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, M * K, K * N, M * N,
                                         batch)
    assert plan["variant_name"] == "TC_GROUPED" and plan["tile_m"] == 32
    sg.sgemm_strided_batched("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, M * K, K * N, M * N, batch)
    assert sg.sgemm_sync_status() == 0
    first = TWO31 // (M * N)
    for b in sorted({0, first - 1, first, first + 1, batch - 2, batch - 1}):
        ref = oracle.sgemm("N", "N", dA[b].cpu().numpy(), dB[b].cpu().numpy(), np.zeros((M, N), np.float32),
                           1.0, 0.0)
        check_exact(dC[b].cpu().numpy(), ref, f"product {b}")
    del dA, dB, dC


@pytest.mark.parametrize("M,N", [(64, 40_000_000), (50_000_000, 48)])
def test_short_side_offsets_beyond_2g(M, N):
    """The short-side kernel with C past 2^31 elements: M short (C written transposed, a column of
    the kernel's tile spans 64 rows of C 40 M floats apart) and N short (rows of 48)."""
    torch = torch_cuda()
    K = 32
    assert M * N > TWO31
    dA, dB = _ints(torch, (M, K), 97), _ints(torch, (K, N), 98)
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    sg.sgemm_set_variant_override("TC_SKINNY", 0)
    try:
        assert sg.sgemm_plan("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)["variant_name"] == "TC_SKINNY"
        sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    if M == 64:
        # every row of columns around the one where row r = 2^31 // N passes 2^31 (offset r * N + c)
        c_b = TWO31 - (TWO31 // N) * N
        cols = sorted({0, 1, N - 2, N - 1, c_b - 1, c_b, c_b + 1, 12_345_678})
        got = dC[:, cols].cpu().numpy()
        ref = oracle.sgemm("N", "N", dA.cpu().numpy(), np.ascontiguousarray(dB[:, cols].cpu().numpy()),
                           np.zeros((M, len(cols)), np.float32), 1.0, 0.0)
    else:
        boundary = TWO31 // N
        rows = sorted({0, boundary - 1, boundary, boundary + 1, M - 2, M - 1, 12345})
        got = dC[rows].cpu().numpy()
        ref = oracle.sgemm("N", "N", dA[rows].cpu().numpy(), dB.cpu().numpy(), np.zeros((len(rows), N), np.float32),
                           1.0, 0.0)
    check_exact(got, ref, f"short side {M}x{N} beyond 2^31")
    del dC
