"""GPU tests of the caller-workspace entry points: sgemm_workspace_size()
reports what the plan needs, sgemm_ex() with that workspace gives the bits
sgemm() gives (the same plan and summation order), rejects a workspace that is
too small or missing without touching C, reuses one workspace in stream order,
and captures into a CUDA graph without memory nodes."""
import numpy as np
import pytest

import oracle
import sgemm_row_major_gb300 as sg
from gpu_util import check_exact, torch_cuda

pytestmark = pytest.mark.gpu


def _dyadic(rng, shape):
    return (rng.integers(-64, 64, size=shape) / 64).astype(np.float32)


def _random(rng, shape):
    return (2 * rng.random(shape) - 1).astype(np.float32)


# (M, N, K, forced variant, forced split): stream-K with shared tiles, several CTAs per tile,
# split-K slices of the FFMA and the any-alignment kernels
SPLITS = [(512, 768, 4096, None, 0), (300, 260, 700, None, 0), (200, 300, 4000, "TMA_128x128", 4),
          (97, 70, 2000, "GENERIC", 3)]


@pytest.mark.parametrize("M,N,K,variant,split", SPLITS, ids=["stream-K", "per-tile split", "ffma split", "generic split"])
def test_ex_matches_sgemm(M, N, K, variant, split):
    torch = torch_cuda()
    rng = np.random.default_rng(M + N + K)
    A, B, C = _random(rng, (M, K)), _random(rng, (K, N)), _random(rng, (M, N))
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    if variant or split:
        sg.sgemm_set_variant_override(variant or "AUTO", split)
    try:
        need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dA, N)
        plan = sg.sgemm_plan("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dA, N)
        assert need == plan["workspace_bytes"] > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        c1 = torch.from_numpy(C).cuda()
        c2 = torch.from_numpy(C).cuda()
        sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, c1, N)
        sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, c2, N, ws, need)
    finally:
        sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status() == 0
    torch.cuda.synchronize()
    check_exact(c2.cpu().numpy(), c1.cpu().numpy(), "sgemm_ex vs sgemm")


def test_ex_rejects_short_or_missing_workspace():
    torch = torch_cuda()
    M, N, K = 512, 768, 4096
    rng = np.random.default_rng(81)
    dA = torch.from_numpy(_random(rng, (M, K))).cuda()
    dB = torch.from_numpy(_random(rng, (K, N))).cuda()
    C = _random(rng, (M, N))
    dC = torch.from_numpy(C).cuda()
    need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dC, N)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dC, N, ws, need - 16, raise_on_error=False) == -15
    assert sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dC, N, None, need, raise_on_error=False) == -14
    assert sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.5, dC, N, ws.data_ptr() + 4, need,
                       raise_on_error=False) == -14
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), C)  # nothing was launched


def test_ex_without_workspace_need():
    """Whole tiles only: no workspace needed, none passed."""
    torch = torch_cuda()
    M, N, K = 128 * 19, 1024, 256
    rng = np.random.default_rng(82)
    A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    assert sg.sgemm_workspace_size("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N) == 0
    sg.sgemm_ex("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N, None, 0)
    assert sg.sgemm_sync_status() == 0
    check_exact(dC.cpu().numpy(), oracle.sgemm("N", "N", A, B, C, 1.5, -0.5), "no workspace")


def test_ex_workspace_reused_in_stream_order():
    """Two calls on one stream share a workspace: the second waits for the first by stream order."""
    torch = torch_cuda()
    M, N, K = 512, 768, 4096
    rng = np.random.default_rng(83)
    mats = [(_dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))) for _ in range(2)]
    dev = [tuple(torch.from_numpy(x).cuda() for x in m) for m in mats]
    need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.0, dev[0][0], K, dev[0][1], N, 1.0, dev[0][2], N)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for dA, dB, dC in dev:
        sg.sgemm_ex("N", "N", M, N, K, 1.0, dA, K, dB, N, 1.0, dC, N, ws, need)
    assert sg.sgemm_sync_status() == 0
    for (A, B, C), (_, _, dC) in zip(mats, dev):
        check_exact(dC.cpu().numpy(), oracle.sgemm("N", "N", A, B, C, 1.0, 1.0), "shared workspace")


def test_ex_graph_capture_replay():
    """A captured sgemm_ex call (stream-K with a fixup launch) replays on new operands."""
    torch = torch_cuda()
    M, N, K = 512, 768, 4096
    dA = torch.empty((M, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((K, N), dtype=torch.float32, device="cuda")
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call():
        sg.sgemm_ex("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N, ws, need)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    rng = np.random.default_rng(84)
    for rep in range(3):
        A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
        dA.copy_(torch.from_numpy(A))
        dB.copy_(torch.from_numpy(B))
        dC.copy_(torch.from_numpy(C))
        g.replay()
        torch.cuda.synchronize()
        assert sg.sgemm_sync_status() == 0
        check_exact(dC.cpu().numpy(), oracle.sgemm("N", "N", A, B, C, 1.5, -0.5), f"replay {rep}")


def test_release_workspace_returns_pool_memory():
    """The pool keeps a large call's split arrays until sgemm_release_workspace() returns them;
    later calls allocate again and give the same bits."""
    torch = torch_cuda()
    M = N = K = 2048
    rng = np.random.default_rng(41)
    A, B = _dyadic(rng, (M, K)), _dyadic(rng, (K, N))
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    assert sg.sgemm_plan("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, dA, N)["workspace_bytes"] >= 64 << 20
    C1 = torch.empty(M, N, device="cuda")
    C2 = torch.empty(M, N, device="cuda")
    sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, C1, N)
    assert sg.sgemm_sync_status() == 0
    free_kept, _ = torch.cuda.mem_get_info()
    sg.sgemm_release_workspace(0)
    free_released, _ = torch.cuda.mem_get_info()
    assert free_released - free_kept >= 60 << 20, (free_kept, free_released)
    sg.sgemm("N", "N", M, N, K, 1.0, dA, K, dB, N, 0.0, C2, N)
    assert sg.sgemm_sync_status() == 0
    assert torch.equal(C1, C2)
    ref = oracle.sgemm("N", "N", A, B)
    check_exact(C2.cpu().numpy(), ref, "after release")
