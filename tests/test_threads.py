"""Calls from host threads other than the one that set up CUDA.

A thread's first CUDA call may be one into the library: it must still find
the device's context (the tensor-map encoder needs one current on the calling
thread).  Calls from several host threads at once, each on its own CUDA stream (ctypes
releases the GIL during the library call): the library's per-device state,
its memory pool and its planner serve them concurrently, and every result
matches the oracle.  Shapes cover whole tiles, stream-K with a fixup and a
workspace from the pool, the caller-workspace entry point and a grouped
batch."""
import threading

import numpy as np
import pytest

import oracle
import sgemm_row_major_gb300 as sg
from gpu_util import check_exact, torch_cuda

pytestmark = pytest.mark.gpu


def _dyadic(rng, shape):
    return (rng.integers(-64, 64, size=shape) / 64).astype(np.float32)


def test_concurrent_calls_from_threads():
    torch = torch_cuda()
    shapes = [(2432, 1024, 256), (512, 768, 4096), (300, 260, 700), (1000, 1300, 700)]
    jobs = []
    for t in range(8):
        M, N, K = shapes[t % len(shapes)]
        rng = np.random.default_rng(100 + t)
        A, B, C = _dyadic(rng, (M, K)), _dyadic(rng, (K, N)), _dyadic(rng, (M, N))
        jobs.append(dict(M=M, N=N, K=K, A=A, B=B, C=C, ex=(t % 2 == 1),
                         dA=torch.from_numpy(A).cuda(), dB=torch.from_numpy(B).cuda(),
                         dC=torch.from_numpy(C).cuda(), stream=torch.cuda.Stream()))
    batch = dict(d=[torch.from_numpy(_dyadic(np.random.default_rng(200), s)).cuda()
                    for s in ((1000, 32, 64), (1000, 64, 48), (1000, 32, 48))], stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    errors = []

    def run(job, reps=20):
        try:
            for _ in range(reps):
                job["dC"].copy_(torch.from_numpy(job["C"]).cuda(), non_blocking=False)
                M, N, K = job["M"], job["N"], job["K"]
                s = job["stream"].cuda_stream
                job["stream"].wait_stream(torch.cuda.current_stream())
                if job["ex"]:
                    need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.5, job["dA"], K, job["dB"], N, -0.5,
                                                   job["dC"], N)
                    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
                    sg.sgemm_ex("N", "N", M, N, K, 1.5, job["dA"], K, job["dB"], N, -0.5, job["dC"], N,
                                ws if need else None, need, s)
                else:
                    sg.sgemm("N", "N", M, N, K, 1.5, job["dA"], K, job["dB"], N, -0.5, job["dC"], N, s)
                torch.cuda.synchronize()
                got = job["dC"].cpu().numpy()
                ref = oracle.sgemm("N", "N", job["A"], job["B"], job["C"], 1.5, -0.5)
                if not np.array_equal(got, ref):
                    errors.append((M, N, K, "mismatch"))
                    return
        except Exception as e:  # reported below
            errors.append(repr(e))

    def run_batch(reps=20):
        try:
            dA, dB, dC = batch["d"]
            for _ in range(reps):
                sg.sgemm_strided_batched("N", "N", 32, 48, 64, 1.0, dA, 64, dB, 48, 0.0, dC, 48, 32 * 64, 64 * 48,
                                         32 * 48, 1000, batch["stream"].cuda_stream)
                batch["stream"].synchronize()
            A, B, C = (x.cpu().numpy() for x in (dA, dB, dC))
            for b in (0, 499, 999):
                ref = oracle.sgemm("N", "N", A[b], B[b], np.zeros((32, 48), np.float32), 1.0, 0.0)
                if not np.array_equal(C[b], ref):
                    errors.append(("batch", b))
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs] + [threading.Thread(target=run_batch)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert sg.sgemm_sync_status() == 0
    assert not errors, errors


@pytest.mark.parametrize("entry", ["sgemm", "sgemm_noalloc", "sgemm_ex", "strided_batched", "sgemm_tf32",
                                   "sgemm_bf16"])
def test_first_cuda_call_of_a_thread(entry):
    """A fresh host thread whose first CUDA call is the library's (stream handle made elsewhere)."""
    torch = torch_cuda()
    rng = np.random.default_rng(7)
    if entry == "strided_batched":
        dims = (300, 32, 48, 64)  # 300 products of 32 x 48 x 64: two to a tensor-core tile on one SM each
    else:
        dims = (1, 640, 384, 512)
    P, M, N, K = dims
    A, B, C = _dyadic(rng, (P, M, K)), _dyadic(rng, (P, K, N)), _dyadic(rng, (P, M, N))
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    need = sg.sgemm_workspace_size("N", "N", M, N, K, 1.5, dA, K, dB, N, -0.5, dC, N) if P == 1 else 0
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    handle = stream.cuda_stream
    out = []

    def run():
        try:
            if entry == "strided_batched":
                out.append(sg.sgemm_strided_batched("N", "N", M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), N, -0.5,
                                                    dC.data_ptr(), N, M * K, K * N, M * N, P, handle))
            elif entry == "sgemm_ex":
                out.append(sg.sgemm_ex("N", "N", M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), N, -0.5,
                                       dC.data_ptr(), N, ws.data_ptr() if need else None, need, handle))
            else:
                fn = getattr(sg, entry)
                out.append(fn("N", "N", M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), N, -0.5, dC.data_ptr(), N,
                              handle))
        except Exception as e:  # reported below
            out.append(repr(e))

    t = threading.Thread(target=run)
    t.start()
    t.join(timeout=120)
    assert not t.is_alive()
    assert out == [0], out
    stream.synchronize()
    got = dC.cpu().numpy()
    ref_fn = getattr(oracle, entry) if entry in ("sgemm_tf32", "sgemm_bf16") else oracle.sgemm
    for b in range(P):
        np.testing.assert_array_equal(got[b], ref_fn("N", "N", A[b], B[b], C[b], 1.5, -0.5))
