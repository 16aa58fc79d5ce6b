"""CUDA-graph capture of the library's calls: a call made on a capturing stream
records its launches (and, for sgemm(), its stream-ordered workspace
allocation), and replaying the graph on new operand values gives the same
results as the oracle.  One eager call per shape comes first: the per-device
set-up (kernel attributes, memory pool, fault word) is not capturable."""
import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import check_exact, torch_cuda

pytestmark = pytest.mark.gpu


def _dyadic(rng, shape):
    return (rng.integers(-64, 64, size=shape) / 64).astype(np.float32)


def _capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("entry", ["sgemm", "sgemm_noalloc"])
def test_single_product_graph_replay(entry):
    """A stream-K shape (GEMM + fixup launch, partial-sum workspace) captured once, replayed on 3 inputs."""
    torch = torch_cuda()
    M, N, K = 512, 768, 4096
    plan = sg.sgemm_plan("N", "N", M, N, K, 1.0, 1 << 20, K, 1 << 20, N, 0.5, 1 << 20, N)
    assert plan["variant_name"] == "TC_TF32X3" and plan["kernel_launches"] == 2
    dA = torch.empty((M, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((K, N), dtype=torch.float32, device="cuda")
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    call = getattr(sg, entry)
    g = _capture(torch, lambda: call("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N))
    rng = np.random.default_rng(61)
    for rep in range(3):
        A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C))
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        check_exact(dC.cpu().numpy(), oracle.sgemm("N", "N", A, B, C, 1.5, -0.5), f"{entry} replay {rep}")


def test_split_operand_graph_replay():
    """The split-operand path (split passes of A and B, GEMM, fixup, and its workspace from the
    pool) captured once and replayed on new inputs."""
    torch = torch_cuda()
    M, N, K = 1280, 1536, 1024
    sg.sgemm_set_variant_override("TC_PRESPLIT", 0)
    try:
        plan = sg.sgemm_plan("N", "T", M, N, K, 1.0, 1 << 20, K, 1 << 20, K, 0.5, 1 << 20, N)
        assert plan["variant_name"] == "TC_PRESPLIT" and plan["kernel_launches"] >= 3
        dA = torch.empty((M, K), dtype=torch.float32, device="cuda")
        dB = torch.empty((N, K), dtype=torch.float32, device="cuda")
        dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        g = _capture(torch, lambda: sg.sgemm("N", "T", M, N, K, 1.5, dA, K, dB, K, -0.5, dC, N))
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    rng = np.random.default_rng(64)
    for rep in range(2):
        A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (N, K)), _dyadic(rng, (M, N))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C))
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        check_exact(dC.cpu().numpy(), oracle.sgemm("N", "T", A, B, C, 1.5, -0.5), f"split-operand replay {rep}")


@pytest.mark.parametrize("entry", ["sgemm_tf32", "sgemm_bf16"])
def test_reduced_precision_graph_replay(entry):
    """The TF32- and BF16-input GEMMs (two rounding passes, the GEMM, the fixup, the workspace
    from the pool) captured once and replayed on new inputs; dyadic values are exact in both
    formats, so the replays equal the oracle bit for bit."""
    torch = torch_cuda()
    M, N, K = 1100, 900, 1500
    dA = torch.empty((K, M), dtype=torch.float32, device="cuda")   # op(A) = A^T
    dB = torch.empty((K, N), dtype=torch.float32, device="cuda")
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    call = getattr(sg, entry)
    g = _capture(torch, lambda: call("T", "N", M, N, K, 1.5, dA, M, dB, N, -0.5, dC, N))
    rng = np.random.default_rng(65)
    ref_fn = getattr(oracle, entry)
    for rep in range(2):
        A, B, C = _dyadic(rng, (K, M)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C))
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        check_exact(dC.cpu().numpy(), ref_fn("T", "N", A, B, C, 1.5, -0.5), f"{entry} replay {rep}")


@pytest.mark.parametrize("M,N", [(64, 2048), (2048, 33)])
def test_short_side_graph_replay(M, N):
    """The short-side path (split pass of the short operand, the GEMM as its programmatic
    dependent, the fixup, workspace from the pool) captured once and replayed on new inputs."""
    torch = torch_cuda()
    K = 3000
    sg.sgemm_set_variant_override("TC_SKINNY", 0)
    try:
        plan = sg.sgemm_plan("N", "N", M, N, K, 1.0, 1 << 20, K, 1 << 20, N, 0.5, 1 << 20, N)
        assert plan["variant_name"] == "TC_SKINNY" and plan["kernel_launches"] == 3
        dA = torch.empty((M, K), dtype=torch.float32, device="cuda")
        dB = torch.empty((K, N), dtype=torch.float32, device="cuda")
        dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        g = _capture(torch, lambda: sg.sgemm("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N))
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    rng = np.random.default_rng(M + N)
    for rep in range(2):
        A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C))
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        check_exact(dC.cpu().numpy(), oracle.sgemm("N", "N", A, B, C, 1.5, -0.5), f"short-side replay {rep}")


def test_graph_replays_back_to_back_accumulate():
    """beta = 1: five replays without a sync between them add op(A) op(B) five times, in order."""
    torch = torch_cuda()
    M, N, K = 300, 260, 700  # stream-K split across several CTAs per tile
    rng = np.random.default_rng(62)
    A, B = _dyadic(rng, (M, K)), _dyadic(rng, (K, N))
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    g = _capture(torch, lambda: sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 1.0, dC, N))
    dC.zero_()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert sg.sgemm_sync_status() == 0
    one = oracle.sgemm("N", "N", A, B, np.zeros((M, N), np.float32), 1.0, 0.0)
    check_exact(dC.cpu().numpy(), (5 * one.astype(np.float64)).astype(np.float32), "5 replays")


@pytest.mark.parametrize("batch,M,N,K,expect", [(1024, 64, 64, 64, "TC_GROUPED"), (16, 256, 384, 512, "TC_TF32X3")])
def test_strided_batch_graph_replay(batch, M, N, K, expect):
    """Strided batches of small products (two to a tensor-core tile) and of large ones, captured and replayed."""
    torch = torch_cuda()
    d = si.make_batched(batch, M, N, K, "N", "T", seed=63, pad=0, gap=0, align=4)
    plan = sg.sgemm_plan_strided_batched("N", "T", M, N, K, 1.0, 1 << 20, d["lda"], 1 << 20, d["ldb"], 0.0,
                                         1 << 20, d["ldc"], d["strideA"], d["strideB"], d["strideC"], batch)
    assert plan["variant_name"] == expect
    dA = torch.empty(d["A"].size, dtype=torch.float32, device="cuda")
    dB = torch.empty(d["B"].size, dtype=torch.float32, device="cuda")
    dC = torch.empty(d["C"].size, dtype=torch.float32, device="cuda")
    g = _capture(torch, lambda: sg.sgemm_strided_batched("N", "T", M, N, K, 2.0, dA, d["lda"], dB, d["ldb"], 0.0,
                                                         dC, d["ldc"], d["strideA"], d["strideB"], d["strideC"],
                                                         batch))
    rng = np.random.default_rng(64)
    for rep in range(2):
        A, B = _dyadic(rng, d["A"].shape), _dyadic(rng, d["B"].shape)
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.fill_(float("nan"))  # beta = 0: C is not read
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        ref = oracle.sgemm_strided_batched("N", "T", M, N, K, 2.0, A, d["lda"], d["strideA"], B, d["ldb"],
                                           d["strideB"], 0.0, np.zeros_like(d["C"]), d["ldc"], d["strideC"], batch)
        check_exact(dC.cpu().numpy(), ref, f"batched {expect} replay {rep}")
