"""sgemm_noalloc: SGEMM for callers that cannot allocate device memory during a call.

sgemm() keeps split-K partial sums in a memory pool that may grow during a
call.  Callers whose own allocator already holds nearly all device memory,
or that cannot afford a pool growing mid-run, use sgemm_noalloc() instead:
it runs the same kernels with the partial sums in a fixed 32 MiB array built
into the library.  These tests call it through the C ABI (ctypes), on shapes
whose plan splits K (so the array is really used), and check its output
against sgemm() on the same inputs for two calls in a row: the second call
finds the array still holding the first call's partial sums.  They also check
that a problem needing more scratch than the array holds is refused with
SGEMM_ERR_SCRATCH_LIMIT and leaves C untouched.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import sgemm_inputs as si
import sgemm_row_major_gb300 as sg

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
SHAPES = [  # (ops, M, N, K, alpha, beta) -- each plan splits K
    ("NN", 1024, 1024, 1024, 1.0, 0.0),
    ("NN", 64, 4096, 16384, 1.0, 0.0),
    ("TN", 300, 500, 3000, 1.5, -0.5),
    ("NT", 200, 130, 4000, -1.0, 1.0),
]


def _c_abi():
    lib = sg.load()
    return lib.sgemm_noalloc


def _stored(op, rows, cols, seed, stream):
    return si.uniform_pm1(*si.stored_shape(op, rows, cols), seed, stream)


@pytest.mark.parametrize("ops,M,N,K,alpha,beta", SHAPES)
def test_noalloc_matches_sgemm_two_calls(ops, M, N, K, alpha, beta):
    import torch
    ta, tb = ops
    A = torch.from_numpy(_stored(ta, M, K, 40 + M, 1)).cuda()
    B = torch.from_numpy(_stored(tb, K, N, 40 + M, 2)).cuda()
    C0 = torch.from_numpy(si.uniform_pm1(M, N, 40 + M, 3)).cuda()
    lda, ldb = A.shape[1], B.shape[1]
    plan = sg.sgemm_plan(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0, N)
    assert plan["split_k"] > 1 and 0 < plan["workspace_bytes"]

    # sgemm_noalloc has no split arrays: where sgemm() splits operands into its workspace, it runs
    # the kernel the planner takes without them, so the reference is sgemm() on that kernel
    fallback = {"TC_SKINNY": "TC_TF32X3", "TC_PRESPLIT": "TC_PAIR"}.get(plan["variant_name"])
    ref = C0.clone()
    if fallback:
        sg.sgemm_set_variant_override(fallback, 0)
    try:
        sg.sgemm(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, ref, N)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0

    # tolerance of the parity tests: |x - y| <= (K + 2) u (|alpha| |op(A)||op(B)| + |beta C|)
    opA = (A.t() if ta == "T" else A).double()
    opB = (B.t() if tb == "T" else B).double()
    S = abs(alpha) * (opA.abs() @ opB.abs()) + abs(beta) * C0.double().abs()
    fn = _c_abi()
    for call in range(2):
        C = C0.clone()
        torch.cuda.synchronize()
        st = fn(ta.encode(), tb.encode(), M, N, K, alpha, A.data_ptr(), lda, B.data_ptr(), ldb, beta,
                C.data_ptr(), N, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream or None))
        assert st == 0, sg.sgemm_status_string(st)
        assert sg.sgemm_sync_status() == 0
        err = (C.double() - ref.double()).abs()
        assert bool((err <= (K + 2) * U * S).all()), f"call {call}: outside the parity tolerance"
        assert torch.equal(C, ref), f"call {call}: differs from sgemm() (same kernels, same order)"


def test_noalloc_refuses_problems_beyond_its_scratch():
    import torch
    M, N, K = 1024, 1024, 8192
    A = torch.ones(M, K, device="cuda")
    B = torch.ones(K, N, device="cuda")
    C = torch.full((M, N), 3.0, device="cuda")
    try:
        sg.sgemm_set_variant_override("TMA_128x128", 9)      # 9 slices x 4 MiB > 32 MiB
        need = sg.sgemm_plan("N", "N", M, N, K, 1.0, A, K, B, N, 0.0, C, N)["workspace_bytes"]
        assert need > sg.NOALLOC_SCRATCH_BYTES
        st = _c_abi()(b"N", b"N", M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N, None)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert st == sg.STATUS["ERR_SCRATCH_LIMIT"]
    assert "SCRATCH_LIMIT" in sg.sgemm_status_string(st)
    torch.cuda.synchronize()
    assert bool((C == 3.0).all()), "a refused call must not touch C"


def test_noalloc_without_split_and_empty_problems():
    import torch
    M, N, K = 2432, 1024, 256      # 152 output tiles (one per SM) and 8 K tiles: no K split
    A = torch.from_numpy(si.uniform_pm1(M, K, 77, 1)).cuda()
    B = torch.from_numpy(si.uniform_pm1(K, N, 77, 2)).cuda()
    assert sg.sgemm_plan("N", "N", M, N, K, 2.0, A, K, B, N, 0.0, A, N)["split_k"] == 1
    ref = torch.empty(M, N, device="cuda")
    out = torch.empty(M, N, device="cuda")
    sg.sgemm("N", "N", M, N, K, 2.0, A, K, B, N, 0.0, ref, N)
    assert sg.sgemm_noalloc("N", "N", M, N, K, 2.0, A, K, B, N, 0.0, out, N) == 0
    assert sg.sgemm_sync_status() == 0
    assert torch.equal(out, ref)
    assert sg.sgemm_noalloc("N", "N", 0, N, K, 1.0, None, K, None, N, 0.0, None, N) == 0
    assert sg.sgemm_noalloc("Q", "N", M, N, K, 1.0, A, K, B, N, 0.0, out, N, raise_on_error=False) == -1
