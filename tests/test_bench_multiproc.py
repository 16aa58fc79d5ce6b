"""CPU tests of the benchmark's multi-replica path (world size 2, gloo on 127.0.0.1).

Each GPU runs an independent replica of the workload (SGEMM shards into
independent problems; no collective touches the data path).  What the ranks
share is the timing: the job time is the slowest replica's, and the job rate
is all replicas' work over that time.  The reference arm runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # replica r took 10 + 5r ms
    ms = bench.reduce_max_ms(local_ms, world)
    out.put((rank, ms, bench.job_tflops(world, 2.0e12, 4, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replica_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tflops in results:
        assert ms == 15.0                                  # the slowest replica
        assert abs(tflops - 2 * 2.0e12 * 4 / 15e-3 / 1e12) < 1e-9


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_ms(7.5, 1) == 7.5
    assert abs(bench.job_tflops(1, 137.4e9, 1, 1.0) - 137.4) < 1e-9   # 137.4 GFLOP in 1 ms


def test_reference_arm_runs_on_rank_zero_only():
    env = {**os.environ, "RANK": "1", "WORLD_SIZE": "2", "OMP_NUM_THREADS": "2"}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--config", "pr1_random", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"] = "0"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--config", "pr1_random", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
