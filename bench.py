"""SGEMM benchmark: TFLOPS (2MNK/t) of libsgemm on the 4096^3 NN workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

One step is one sgemm() call over the whole problem (C = 1.5*A*B - 0.5*C at
4096^3 by default).  Prints ONE JSON line (rank 0).  Timing: W untimed
warm-up steps, then exactly K steps between a barrier + device synchronise
on both sides; per-step CUDA events on the launching stream give the kernel
time for the roofline.  Two input sets of 192 MiB are used in turn, so every
step reads inputs larger than the 129 MB L2 (no flush kernel).

``e2e``: the same metric through the C ABI with host buffers: every step is
one sgemm_host() call on pinned host A, B, C (it copies B, streams op(A) and C
in row blocks overlapping the GEMM, and writes C back to host memory).

``--impl reference``: the CPU oracle (plain triple loop, double accumulation)
timed on this machine's host cores on a bounded sample of rows of the same
workload, scaled to TFLOPS.  Under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import sgemm_inputs as si  # noqa: E402

METRIC = "SGEMM TFLOPS (2MNK/t) at 4096^3 NN on 1 GB300; % of FP32 FFMA peak"
UNIT = "TFLOPS"
FMA_PER_SM_PER_CLK = 128  # FP32 FMA lanes per SM (4 sub-partitions x 32)
# per-launch DRAM traffic of the dominant kernel by (variant, workload), from ncu captures
# (profiles/traffic.json, written with the summaries in profiles/); reported while the kernel's
# source digest still matches the one the capture was taken with
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# dense tensor-core peaks (PFLOP/s, nominal) used to scale the measured bf16 peak to tf32
NOMINAL_BF16_PF, NOMINAL_TF32_PF = 2.25, 1.1
TF32_PRODUCTS = 3  # tensor-core products per useful FMA in the 3xTF32 split
# entry points bench.py can time: (library function, plan function, oracle function, dtype)
ENTRIES = {"sgemm": ("sgemm", "sgemm_plan", "sgemm", "f32"),
           "tf32": ("sgemm_tf32", "sgemm_tf32_plan", "sgemm_tf32", "tf32 inputs, f32 accumulation"),
           "bf16": ("sgemm_bf16", "sgemm_bf16_plan", "sgemm_bf16", "bf16 inputs, f32 accumulation")}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=si.HEADLINE,
                    help="workload name from sgemm_inputs.CASES or sgemm_inputs.BATCHED_CASES")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prewarm-s", type=float, default=0.5, help="untimed seconds of steps before the warm-up")
    ap.add_argument("--variant", default="AUTO", help="planner override (tests and experiments)")
    ap.add_argument("--split", type=int, default=0,
                    help="planner override of the K split (0 = planner's choice; with the tensor-core kernel, "
                         "1 = one CTA per output tile, hardware-scheduled)")
    ap.add_argument("--entry", choices=list(ENTRIES), default="sgemm",
                    help="entry point timed: sgemm (the FP32 contract) or the reduced-precision-input GEMMs "
                         "sgemm_tf32 / sgemm_bf16 (inputs rounded to TF32 / BF16, FP32 accumulation)")
    ap.add_argument("--no-cublas-context", action="store_true",
                    help="skip the cuBLAS FP32 context number (torch.matmul, TF32 off)")
    return ap.parse_args()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons in the background."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu_id = gpu_id
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", str(self.period_ms)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [l.split(", ") for (t, l) in self.lines if t0 <= t <= t1]
        rows = [r for r in rows if len(r) == len(self.FIELDS)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the loaded window"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        power = [float(r[3]) for r in rows if re.match(r"^[0-9.]+$", r[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def gpu_selector(device_index: int) -> str:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        if uuid and uuid != "None":
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    if device_index < len(parts) and parts[device_index].strip().isdigit():
        return parts[device_index].strip()
    return str(device_index)


# ---------------------------------------------------------------- helpers

def traffic_from_profile(variant: str, workload: str, digest: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu capture record, if it is
    current (same kernel source digest)."""
    try:
        entries = json.load(open(TRAFFIC_FILE))["entries"]
    except (OSError, ValueError, KeyError):
        return None
    for e in entries:
        if e.get("variant") == variant and e.get("workload") == workload and e.get("kernel_digest") == digest:
            return int(e["traffic_bytes_per_launch"])
    return None


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


def oracle_sample_run(case, d, rows, entry="sgemm"):
    """Oracle (the entry point's oracle function) on `rows` of C; returns seconds."""
    import oracle
    fn = getattr(oracle, ENTRIES[entry][2])
    from_rows = np.asarray(rows, dtype=np.int64)
    A = d["A"][:, :(case.M if case.transA == "T" else case.K)]
    A = np.ascontiguousarray(A[:, from_rows] if case.transA == "T" else A[from_rows, :])
    B = d["B"][:, :(case.K if case.transB == "T" else case.N)]
    C = np.ascontiguousarray(d["C"][from_rows, :case.N])
    t0 = time.perf_counter()
    fn(case.transA, case.transB, A, B, C, case.alpha, case.beta, M=len(from_rows), N=case.N, K=case.K)
    return time.perf_counter() - t0


def cpu_rows_for(case, d, seconds: float, entry="sgemm"):
    """Rows of C whose oracle run takes about `seconds` (calibrated on a few rows)."""
    probe = list(range(min(4, case.M)))
    t = max(oracle_sample_run(case, d, probe, entry), 1e-4)
    n = int(max(1, min(case.M, round(len(probe) * seconds / t))))
    return list(range(n))


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def cpu_baseline(case, d, seconds, entry="sgemm"):
    import oracle
    cores = oracle.num_threads()
    rows = cpu_rows_for(case, d, seconds, entry)
    t = oracle_sample_run(case, d, rows, entry)
    flops = si.flops(len(rows), case.N, case.K)
    out = {"value": flops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{len(rows)} of {case.M} rows of C ({len(rows)}x{case.N}x{case.K}, "
                     f"{flops / 1e9:.2f} GFLOP) in {t:.1f} s; TFLOPS = 2*rows*N*K/t",
           "cpu": cpu_model()}
    # the same oracle on one core, for a per-core figure
    oracle.set_num_threads(1)
    try:
        rows1 = cpu_rows_for(case, d, min(3.0, seconds / 4), entry)
        t1 = oracle_sample_run(case, d, rows1, entry)
        out["per_core"] = {"value": si.flops(len(rows1), case.N, case.K) / t1 / 1e12, "unit": UNIT,
                           "sample": f"{len(rows1)} rows in {t1:.2f} s on 1 thread"}
    finally:
        oracle.set_num_threads(cores)
    return out


def reduce_max_ms(ms: float, world: int, device=None) -> float:
    """Slowest rank's time: the job is done when every replica is done."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Whole-job rate: the work all replicas did over the slowest replica's time."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    case = si.case(args.config)
    d = si.make_case(case)
    import oracle
    oracle.build()
    per_step = max(0.5, min(5.0, 100.0 / max(1, args.steps + args.warmup)))
    rows = cpu_rows_for(case, d, per_step)
    for _ in range(args.warmup):
        oracle_sample_run(case, d, rows)
    times = [oracle_sample_run(case, d, rows) for _ in range(args.steps)]
    total = sum(times)
    flops = si.flops(len(rows), case.N, case.K) * args.steps
    value = flops / total / 1e12
    sample = (f"each step: {len(rows)} of {case.M} rows of C ({len(rows)}x{case.N}x{case.K}); "
              f"TFLOPS = 2*rows*N*K/t")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate",
        "data": "synthetic", "config": config_block(case, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(case, n_gpus, entry=None):
    """The workload; `entry` names a reduced-precision-input entry point when that is what runs."""
    out = {"workload": f"sgemm_{case.transA}{case.transB}_{case.M}x{case.N}x{case.K}",
           "name": case.name, "M": case.M, "N": case.N, "K": case.K, "ops": case.ops,
           "alpha": case.alpha, "beta": case.beta, "inputs": case.dist, "layout": "row-major fp32",
           "parallelism": f"replicas x{n_gpus}"}
    if entry:
        out["entry"] = entry
    return out


# ---------------------------------------------------------------- our arm

def cublas_context(case, sets, steps, stream, entry="sgemm"):
    """cuBLAS through torch.addmm on the same shapes and input sets, as a context number: FP32
    SGEMM with TF32 disabled (entry "sgemm"); with TF32 enabled (entry "tf32"); or on inputs cast
    to BF16 inside the timed region, BF16 output (entry "bf16").  Computes
    alpha*op(A)@op(B) + beta*C into a preallocated output; not part of the measured path.
    """
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = entry == "tf32"
    try:
        dt = torch.bfloat16 if entry == "bf16" else torch.float32
        outs = [torch.empty(case.M, case.N, dtype=dt, device=s[2].device) for s in sets]

        def one(i):
            A, B, C = sets[i & 1]
            a = A[:, :(case.M if case.transA == "T" else case.K)]
            b = B[:, :(case.K if case.transB == "T" else case.N)]
            a = a.t() if case.transA == "T" else a
            b = b.t() if case.transB == "T" else b
            c = C[:, :case.N]
            if entry == "bf16":
                a, b, c = a.to(dt), b.to(dt), c.to(dt)
            torch.addmm(c, a, b, beta=case.beta, alpha=case.alpha, out=outs[i & 1])

        for i in range(5):
            one(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            one(i)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        what = {"sgemm": "cuBLAS FP32 via torch.addmm, allow_tf32=False",
                "tf32": "cuBLAS TF32 via torch.addmm, allow_tf32=True",
                "bf16": "cuBLAS BF16 via torch.addmm on A, B, C cast to BF16 in the timed region, BF16 output"}[entry]
        return {"value": si.flops(case.M, case.N, case.K) / (ms * 1e-3) / 1e12, "unit": UNIT,
                "what": what + ", same shapes and input sets; context only"}
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


L2_BYTES = 129 * 1000 * 1000  # GB300 L2


def l2_flusher(dev, set_bytes):
    """A step-separating L2 flush (a memset of 2x the L2 size) when one input set fits in L2, else None."""
    import torch
    if set_bytes >= L2_BYTES:
        return None
    buf = torch.empty(2 * L2_BYTES + (1 << 20), dtype=torch.uint8, device=dev)
    state = {"v": 0}

    def flush():
        state["v"] = (state["v"] + 1) & 0xFF
        buf.fill_(state["v"])
    return flush


def snapshot_mhz(before, after):
    """Median over SMs of (cycle counter delta) / (global timer delta) between two per-SM clock
    snapshots (sgemm_clock_snapshot), in MHz, and the number of SMs it covers."""
    b = before.view(-1, 2).cpu().numpy().astype(np.int64)
    a = after.view(-1, 2).cpu().numpy().astype(np.int64)
    ok = (b[:, 1] > 0) & (a[:, 1] > b[:, 1]) & (a[:, 0] > b[:, 0])
    if not ok.any():
        return None, 0
    mhz = (a[ok, 0] - b[ok, 0]) / (a[ok, 1] - b[ok, 1]) * 1e3
    return float(np.median(mhz)), int(ok.sum())


def timed_steps(step, args, stream, dev, local, barrier, world, flush=None):
    """Pre-warm, W warm-up steps, then exactly K timed steps between barriers.

    With `flush`, L2 is flushed before every step (outside the step's events)
    and the job time is the sum of the steps' event times.  Clocks: nvidia-smi
    samples every 50 ms from the start of the pre-warm to the end of the timed
    steps (the loaded window: a timed region of a few ms holds no sample of its
    own), and a per-SM clock snapshot just before the first and just after the
    last timed step gives the SMs' average clock over exactly the timed steps.
    Returns (per-step ms from CUDA events on `stream`, the slowest rank's job
    ms, the clock record)."""
    import torch
    import sgemm_row_major_gb300 as sg
    sampler = ClockSampler(gpu_selector(local))
    sampler.start()
    time.sleep(0.2)
    t_load = time.time()
    t_end = time.time() + args.prewarm_s
    i = 0
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 20 == 0:
            torch.cuda.synchronize(dev)
    for w in range(args.warmup):
        step(w)
    barrier()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    snaps = [torch.zeros(2 * 1024, dtype=torch.int64, device=dev) for _ in range(2)]
    barrier()
    t0_wall = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    sg.sgemm_clock_snapshot(snaps[0], stream)
    g0.record(stream)
    for s in range(args.steps):
        if flush:
            flush()
        ev[s][0].record(stream)
        step(s)
        ev[s][1].record(stream)
    g1.record(stream)
    sg.sgemm_clock_snapshot(snaps[1], stream)
    barrier()
    t1_wall = time.time()
    time.sleep(0.1)
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    job_ms = sum(step_ms) if flush else g0.elapsed_time(g1)
    total_ms = reduce_max_ms(job_ms, world, dev)
    clocks = sampler.summary(t_load, t1_wall)
    clocks["window"] = (f"nvidia-smi every 50 ms over the loaded window: pre-warm {args.prewarm_s:.1f} s, "
                        f"{args.warmup} warm-up and {args.steps} timed steps ({1e3 * (t1_wall - t_load):.0f} ms)")
    clocks["timed_samples"] = len([1 for (t, _) in sampler.lines if t0_wall <= t <= t1_wall])
    mhz, n_sms = snapshot_mhz(*snaps)
    clocks["sm_mhz_timed_steps"] = mhz
    clocks["sm_mhz_timed_steps_basis"] = (f"median over {n_sms} SMs of SM cycle-counter / global-timer deltas "
                                          f"between snapshots just before and just after the timed steps")
    return step_ms, total_ms, clocks


def l2_hot_ms(step, args, stream, dev, barrier, world):
    """For inputs that fit in L2 (timed flushed above): the same K steps back to back on one input
    set, with no flush, so its operands stay in L2.  Returns the slowest rank's ms per step."""
    import torch
    for w in range(max(1, args.warmup)):
        step(0)
    barrier()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step(0)
    g1.record(stream)
    barrier()
    return reduce_max_ms(g0.elapsed_time(g1), world, dev) / args.steps


def l2_hot_block(flush, hot_ms, flops_step):
    if not flush:
        return {"value": None, "note": "one input set is larger than the 129 MB L2: no L2-hot timing"}
    return {"value": flops_step / (hot_ms * 1e-3) / 1e12, "unit": "TFLOPS", "ms_per_step": hot_ms,
            "note": "the same steps back to back on one input set, no L2 flush (operands L2-resident)"}


def step_stats(step_ms):
    return {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)}


def l2_note(flush):
    return ("L2 flushed before every step (2x L2 memset outside the step's events); value from the "
            "steps' event times" if flush else
            "two input sets used in turn, each larger than the 129 MB L2; no flush")


KERNEL_NAMES = {
    "TC_TF32X3": "tf32x3_gemm_kernel (tcgen05.mma kind::tf32, 3xTF32 split)",
    "TC_PAIR": "pair_gemm_kernel (tcgen05.mma cta_group::2 kind::tf32, 3xTF32 split, 256x128 tiles on CTA pairs)",
    "TC_PRESPLIT": "presplit_gemm_kernel (tcgen05.mma cta_group::2 kind::tf32, both operands from shared memory, "
                   "256x256 tiles on CTA pairs) after split_rows/split_transpose (A and B split once into TF32 hi "
                   "and FP32 lo)",
    "TC_SKINNY": "skinny_gemm_kernel (tcgen05.mma kind::tf32 N=64, 3xTF32 split, 128 x 64 tiles along the long x "
                 "short side) after split_rows/split_transpose of the short operand",
}


def kernel_digest(lib_build, variant):
    """Source digest of the kernel a variant runs (matches the digest in its committed profile)."""
    if variant == "TC_PRESPLIT":
        return lib_build.presplit_kernel_digest()
    if variant == "TC_PAIR":
        return lib_build.pair_kernel_digest()
    if variant in ("TC_TF32X3", "TC_GROUPED"):
        return lib_build.tc_kernel_digest()
    if variant == "SMALL":
        return lib_build.small_kernel_digest()
    if variant == "TC_SKINNY":
        return lib_build.skinny_kernel_digest()
    return lib_build.tma_kernel_digest()


def tensor_roofline(achieved, peaks, traffic, kernel_ms, variant="TC_TF32X3"):
    """Roofline object of the 3xTF32 tensor-core kernels (see the module docstrings of the kernels)."""
    bf16 = peaks.get("bf16_tflops")
    basis = "measured" if bf16 else "fallback"
    bf16 = bf16 or 1900.0
    tf32 = bf16 * NOMINAL_TF32_PF / NOMINAL_BF16_PF
    return {"bound": "tensor", "achieved": achieved, "peak": tf32 / TF32_PRODUCTS, "unit": "TFLOP/s",
            "frac": achieved / (tf32 / TF32_PRODUCTS), "traffic": traffic,
            "peak_basis": f"{basis} bf16 burst {bf16:.0f} TFLOP/s x nominal tf32/bf16 "
                          f"{NOMINAL_TF32_PF}/{NOMINAL_BF16_PF} = {tf32:.0f} TFLOP/s of tf32, / {TF32_PRODUCTS} "
                          f"tensor products per SGEMM FMA (3xTF32 split); achieved counts 2MNK only",
            "kernel": KERNEL_NAMES.get(variant, KERNEL_NAMES["TC_TF32X3"]), "kernel_ms": kernel_ms,
            "kernel_ms_covers": ("one sgemm() call: the split passes of A and B, the GEMM kernel and, when "
                                 "stream-K tiles are shared, the fixup kernel" if variant == "TC_PRESPLIT" else
                                 "one sgemm() call: the split pass of the short operand, the GEMM kernel and, "
                                 "when stream-K tiles are shared, the fixup kernel" if variant == "TC_SKINNY" else
                                 "one sgemm() call: the GEMM kernel and, when stream-K tiles are shared, "
                                 "the fixup kernel after it")}


def reduced_roofline(achieved, peaks, variant, kernel_ms, traffic):
    """Roofline object of the reduced-precision-input GEMMs (one tensor-core product per term):
    the measured bf16 peak for BF16 inputs, that peak x the nominal tf32/bf16 ratio for TF32."""
    bf16 = peaks.get("bf16_tflops")
    basis = "measured" if bf16 else "fallback"
    bf16 = bf16 or 1900.0
    bf = variant == "TC_BF16"
    peak = bf16 if bf else bf16 * NOMINAL_TF32_PF / NOMINAL_BF16_PF
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic,
            "peak_basis": f"{basis} bf16 burst {bf16:.0f} TFLOP/s" +
                          ("" if bf else f" x nominal tf32/bf16 {NOMINAL_TF32_PF}/{NOMINAL_BF16_PF}") +
                          "; one tensor-core product per term; achieved counts 2MNK only",
            "kernel": ("presplit_gemm_kernel<1, BF16> (tcgen05.mma cta_group::2 kind::f16, 256x256 tiles, 64-deep K "
                       "tiles)" if bf else "presplit_gemm_kernel<1> (tcgen05.mma cta_group::2 kind::tf32, 256x256 "
                       "tiles)") + " after the rounding passes of A and B",
            "kernel_ms": kernel_ms,
            "kernel_ms_covers": "one call: the rounding passes of A and B, the GEMM kernel and, when stream-K "
                                "tiles are shared, the fixup kernel"}


def hbm_bound_roofline(roof, nbytes, flops_step, kernel_ms, peaks):
    """Switches a tensor-core roofline to the HBM roof when the call's algorithmic bytes take longer
    at the measured HBM bandwidth than its FLOPs at the tensor peak (the tensor figures stay
    beside it)."""
    hbm = peaks.get("hbm_gbs")
    hbm_basis = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    roof["algorithmic_bytes"] = nbytes
    if nbytes / (hbm * 1e9) > flops_step / (roof["peak"] * 1e12):
        gbs = nbytes / (kernel_ms * 1e-3) / 1e9
        tensor = {k: roof[k] for k in ("achieved", "peak", "unit", "frac", "peak_basis")}
        roof.update({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_basis": f"{hbm_basis} HBM copy bandwidth", "tensor": tensor})
    return roof


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sgemm_row_major_gb300 import build as lib_build
    lib_build.build()
    import sgemm_row_major_gb300 as sg

    case = si.case(args.config)
    d = si.make_case(case)
    M, N, K = case.M, case.N, case.K
    stream = torch.cuda.current_stream(dev)
    if args.variant != "AUTO" or args.split:
        sg.sgemm_set_variant_override(args.variant, args.split)
    sh = stream.cuda_stream

    # two device-resident input sets, used in turn
    sets = []
    for _ in range(2):
        sets.append(tuple(torch.from_numpy(d[k]).to(dev) for k in ("A", "B", "C")))
    torch.cuda.synchronize(dev)

    lib_fn, plan_fn, _, dtype = ENTRIES[args.entry]
    call = getattr(sg, lib_fn)
    plan = getattr(sg, plan_fn)(case.transA, case.transB, M, N, K, case.alpha, sets[0][0], d["lda"], sets[0][1],
                                d["ldb"], case.beta, sets[0][2], d["ldc"])

    def step(i):
        A, B, C = sets[i & 1]
        call(case.transA, case.transB, M, N, K, case.alpha, A, d["lda"], B, d["ldb"], case.beta, C, d["ldc"], sh)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    flush = l2_flusher(dev, sum(x.numel() * 4 for x in sets[0]))
    step_ms, total_ms, clocks = timed_steps(step, args, stream, dev, local, barrier, world, flush)
    hot_ms = l2_hot_ms(step, args, stream, dev, barrier, world) if flush else None
    if sg.sgemm_sync_status(sh) != 0:
        raise RuntimeError("libsgemm reported a kernel fault during the benchmark")
    flops_step = si.flops(M, N, K)
    value = job_tflops(world, flops_step, args.steps, total_ms)
    kernel_ms = statistics.mean(step_ms)
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12

    # ---- e2e: host buffers through the C ABI (sgemm_host), copies inside the timed region
    hA, hB, hC = (torch.from_numpy(d[k]).pin_memory() for k in ("A", "B", "C"))

    if args.entry != "sgemm":
        # no host-buffer form of the reduced-precision entry points: the same copies, made here
        dA, dB, dC = (torch.empty_like(x) for x in sets[0])

        def e2e_step():
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            if case.beta != 0.0:
                dC.copy_(hC, non_blocking=True)
            call(case.transA, case.transB, M, N, K, case.alpha, dA, d["lda"], dB, d["ldb"], case.beta, dC,
                 d["ldc"], sh)
            hC.copy_(dC, non_blocking=True)
    else:
        def e2e_step():
            sg.sgemm_host(case.transA, case.transB, M, N, K, case.alpha, hA, d["lda"], hB, d["ldb"], case.beta,
                          hC, d["ldc"], sh)

    for _ in range(2 if args.e2e_steps > 0 else 0):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = reduce_max_ms(e0.elapsed_time(e1), world, dev)
    e2e_value = job_tflops(world, flops_step, args.e2e_steps, e2e_ms) if args.e2e_steps > 0 else None
    h2d = (hA.numel() + hB.numel() + (hC.numel() if case.beta != 0.0 else 0)) * 4
    d2h = hC.numel() * 4

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    peaks = measured_peaks()
    max_mhz = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    ffma_peak = sms * FMA_PER_SM_PER_CLK * 2 * max_mhz * 1e6 / 1e12
    variant = plan["variant_name"]
    if variant in ("TC_TF32", "TC_BF16"):
        roof = reduced_roofline(achieved, peaks, variant, kernel_ms,
                                traffic_from_profile(variant, case.name, lib_build.presplit_kernel_digest()))
        hbm_bound_roofline(roof, si.min_bytes(M, N, K, case.beta), flops_step, kernel_ms, peaks)
    elif variant in ("TC_TF32X3", "TC_PAIR", "TC_PRESPLIT", "TC_SKINNY"):
        roof = tensor_roofline(achieved, peaks,
                               traffic_from_profile(variant, case.name, kernel_digest(lib_build, variant)),
                               kernel_ms, variant)
        hbm_bound_roofline(roof, si.min_bytes(M, N, K, case.beta), flops_step, kernel_ms, peaks)
    else:
        roof = {"bound": "alu", "achieved": achieved, "peak": ffma_peak, "unit": "TFLOP/s",
                "frac": achieved / ffma_peak,
                "traffic": traffic_from_profile(variant, case.name, lib_build.tma_kernel_digest()),
                "peak_basis": f"{sms} SMs x {FMA_PER_SM_PER_CLK} FP32 FMA/clk x 2 FLOP x {max_mhz:.0f} MHz max SM clock",
                "kernel": "tma_gemm_kernel (SIMT FFMA2)" if variant.startswith("TMA") else variant,
                "kernel_ms": kernel_ms}
        if clocks.get("sm_mhz"):
            roof["frac_at_sampled_clock"] = achieved / (sms * FMA_PER_SM_PER_CLK * 2 * clocks["sm_mhz"] * 1e6 / 1e12)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "step_ms": step_stats(step_ms),
        "config": config_block(case, world, None if args.entry == "sgemm" else lib_fn),
        "l2_hot": l2_hot_block(flush, hot_ms, flops_step),
        "run": {"l2": l2_note(flush), "prewarm_s": args.prewarm_s,
                "plan": {k: plan[k] for k in ("variant_name", "tile_m", "tile_n", "tile_k", "stages",
                                              "split_k", "grid_x", "grid_y", "dp_tiles", "sk_tiles",
                                              "kernel_launches")}},
        "pct_ffma_peak": 100.0 * achieved / ffma_peak,
        "ffma_peak": {"value": ffma_peak, "unit": "TFLOP/s",
                      "basis": f"{sms} SMs x {FMA_PER_SM_PER_CLK} FP32 FMA/clk x 2 FLOP x {max_mhz:.0f} MHz"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": plan["kernel_launches"] * args.steps,
        "clocks": clocks,
    }
    if not args.no_cublas_context:
        line["context_cublas_fp32"] = cublas_context(case, sets, min(args.steps, 50), stream)
        if args.entry != "sgemm":
            line["context_cublas_" + args.entry] = cublas_context(case, sets, min(args.steps, 50), stream,
                                                                  args.entry)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, d, args.cpu_seconds, args.entry)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- strided batch workloads

BATCHED_METRIC = "strided-batched SGEMM TFLOPS (2*batch*MNK/t) on 1 GB300"


def batched_config_block(c, d, n_gpus):
    return {"workload": f"sgemm_strided_batched_{c.transA}{c.transB}_{c.batch}x{c.M}x{c.N}x{c.K}",
            "name": c.name, "batch": c.batch, "M": c.M, "N": c.N, "K": c.K, "ops": c.ops,
            "alpha": c.alpha, "beta": c.beta, "inputs": c.dist, "shared": c.shared or "none",
            "strides": {k: d["stride" + k] for k in "ABC"}, "layout": "row-major fp32, packed products",
            "parallelism": f"replicas x{n_gpus}"}


def batched_oracle_run(c, d, products):
    """Oracle strided batch over the first `products` products; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.sgemm_strided_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, d["A"], d["lda"], d["strideA"],
                                 d["B"], d["ldb"], d["strideB"], c.beta, d["C"], d["ldc"], d["strideC"], products)
    return time.perf_counter() - t0


def batched_oracle_sample(c, d, seconds):
    """Number of whole products whose oracle run takes about `seconds`, and that run's time."""
    t = max(batched_oracle_run(c, d, 1), 1e-4)
    n = int(max(1, min(c.batch, round(seconds / t))))
    return n, batched_oracle_run(c, d, n)


def run_reference_batched(args, c):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    d = si.make_batched(c.batch, c.M, c.N, c.K, c.transA, c.transB, seed=c.seed, dist=c.dist, shared=c.shared,
                        c_init="uniform" if c.beta != 0 else "zero")
    per_step = max(0.5, min(5.0, 100.0 / max(1, args.steps + args.warmup)))
    products, _ = batched_oracle_sample(c, d, per_step)
    for _ in range(args.warmup):
        batched_oracle_run(c, d, products)
    total = sum(batched_oracle_run(c, d, products) for _ in range(args.steps))
    value = products * si.flops(c.M, c.N, c.K) * args.steps / total / 1e12
    sample = (f"each step: the first {products} of {c.batch} products ({c.M}x{c.N}x{c.K} each); "
              f"TFLOPS = 2*products*M*N*K/t")
    print(json.dumps({
        "impl": "reference", "metric": BATCHED_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate",
        "data": "synthetic", "config": batched_config_block(c, d, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def batched_bytes(c):
    """Algorithmic bytes of one strided-batch call: each operand read once (a shared one once in all),
    C written once, and read too when beta != 0."""
    n_a = 1 if "A" in c.shared else c.batch
    n_b = 1 if "B" in c.shared else c.batch
    return 4 * (n_a * c.M * c.K + n_b * c.K * c.N + c.batch * c.M * c.N * (2 if c.beta != 0 else 1))


def batched_roofline(c, plan, flops_step, achieved, kernel_ms, peaks, dev, lib_build):
    """Roofline object of the kernel a strided batch ran on.  For the tensor-core kernel the bound is
    whichever of the 3xTF32 tensor peak and HBM takes longer for the call's algorithmic work."""
    variant = plan["variant_name"]
    if variant in ("TC_TF32X3", "TC_GROUPED", "TC_PAIR", "TC_PRESPLIT"):
        traffic = traffic_from_profile(variant, c.name, kernel_digest(lib_build, variant))
        roof = tensor_roofline(achieved, peaks, traffic, kernel_ms, variant)
        if variant == "TC_GROUPED":
            group = 128 // plan["tile_m"]
            tiles = (c.batch + group - 1) // group
            roof["kernel"] = f"tf32x3_gemm_kernel, {group} products per 128x128 tile (block-diagonal)"
            roof["useful_fraction_of_tensor_work"] = c.batch * c.M * c.N / (tiles * 128 * 128)
        return hbm_bound_roofline(roof, batched_bytes(c), flops_step, kernel_ms, peaks)
    if variant == "SMALL":
        return small_roofline(c, flops_step, kernel_ms, peaks, dev,
                              traffic_from_profile(variant, c.name, lib_build.small_kernel_digest()))
    return {"bound": "alu", "achieved": achieved, "peak": None, "unit": "TFLOP/s", "frac": None,
            "traffic": None, "kernel": variant, "kernel_ms": kernel_ms}


def small_roofline(c, flops_step, kernel_ms, peaks, dev, traffic):
    """Roofline of the small-product kernel: each operand is read once and C written once (read too
    when beta != 0), so the launch is bound by HBM or by the FP32 FMA pipes, whichever takes longer."""
    import torch
    nbytes = batched_bytes(c)
    hbm = peaks.get("hbm_gbs")
    hbm_basis = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = peaks.get("sm_max_mhz") or 2070.0
    ffma_peak = sms * FMA_PER_SM_PER_CLK * 2 * max_mhz * 1e6 / 1e12
    t = kernel_ms * 1e-3
    gbs, tflops = nbytes / t / 1e9, flops_step / t / 1e12
    hbm_bound = nbytes / (hbm * 1e9) >= flops_step / (ffma_peak * 1e12)
    out = {"kernel": "small_gemm_kernel (persistent, a 64x64 tile per product, SIMT FFMA2)", "kernel_ms": kernel_ms,
           "traffic": traffic, "algorithmic_bytes": nbytes,
           "alu": {"achieved": tflops, "peak": ffma_peak, "unit": "TFLOP/s", "frac": tflops / ffma_peak},
           "hbm": {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "basis": hbm_basis}}
    if hbm_bound:
        out.update({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm})
    else:
        out.update({"bound": "alu", "achieved": tflops, "peak": ffma_peak, "unit": "TFLOP/s",
                    "frac": tflops / ffma_peak})
    return out


def run_ours_batched(args, c):
    """One step = one sgemm_strided_batched() call over the whole batch."""
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from sgemm_row_major_gb300 import build as lib_build
    lib_build.build()
    import sgemm_row_major_gb300 as sg

    d = si.make_batched(c.batch, c.M, c.N, c.K, c.transA, c.transB, seed=c.seed, dist=c.dist, shared=c.shared,
                        c_init="uniform" if c.beta != 0 else "zero")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    if args.variant != "AUTO" or args.split:
        sg.sgemm_set_variant_override(args.variant, args.split)
    sets = [tuple(torch.from_numpy(d[k]).to(dev) for k in ("A", "B", "C")) for _ in range(2)]
    torch.cuda.synchronize(dev)
    strides = (d["strideA"], d["strideB"], d["strideC"])
    plan = sg.sgemm_plan_strided_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, sets[0][0], d["lda"],
                                         sets[0][1], d["ldb"], c.beta, sets[0][2], d["ldc"], *strides, c.batch)

    def step(i):
        A, B, C = sets[i & 1]
        sg.sgemm_strided_batched(c.transA, c.transB, c.M, c.N, c.K, c.alpha, A, d["lda"], B, d["ldb"], c.beta, C,
                                 d["ldc"], *strides, c.batch, sh)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    flush = l2_flusher(dev, sum(x.numel() * 4 for x in sets[0]))
    step_ms, total_ms, clocks = timed_steps(step, args, stream, dev, local, barrier, world, flush)
    hot_ms = l2_hot_ms(step, args, stream, dev, barrier, world) if flush else None
    if sg.sgemm_sync_status(sh) != 0:
        raise RuntimeError("libsgemm reported a kernel fault during the benchmark")
    flops_step = c.batch * si.flops(c.M, c.N, c.K)
    value = job_tflops(world, flops_step, args.steps, total_ms)
    kernel_ms = statistics.mean(step_ms)
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks = measured_peaks()
    line = {
        "metric": BATCHED_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "step_ms": step_stats(step_ms),
        "config": batched_config_block(c, d, world),
        "l2_hot": l2_hot_block(flush, hot_ms, flops_step),
        "run": {"l2": l2_note(flush), "prewarm_s": args.prewarm_s,
                "plan": {k: plan[k] for k in ("variant_name", "tile_m", "tile_n", "split_k", "grid_x", "grid_y",
                                              "dp_tiles", "sk_tiles", "kernel_launches")}},
        "roofline": batched_roofline(c, plan, flops_step, achieved, kernel_ms, peaks, dev, lib_build),
        "e2e": {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "note": "no host-buffer batched entry point; the device-resident value is the measurement"},
        "gpu_launches": plan["kernel_launches"] * args.steps,
        "clocks": clocks,
    }
    if not args.no_cublas_context:
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        try:
            def view(flat, n, rows, cols, ld, stride):
                return flat.as_strided((n, rows, cols), (stride, ld, 1))
            outs = [torch.empty_like(s_[2]) for s_ in sets]

            def one(i):
                A, B, C = sets[i & 1]
                ar, ac = si.stored_shape(c.transA, c.M, c.K)
                br, bc = si.stored_shape(c.transB, c.K, c.N)
                a = view(A, c.batch, ar, ac, d["lda"], d["strideA"])
                b = view(B, c.batch, br, bc, d["ldb"], d["strideB"])
                a = a.transpose(1, 2) if c.transA == "T" else a
                b = b.transpose(1, 2) if c.transB == "T" else b
                o = view(outs[i & 1], c.batch, c.M, c.N, d["ldc"], d["strideC"])
                torch.baddbmm(view(C, c.batch, c.M, c.N, d["ldc"], d["strideC"]), a, b, beta=c.beta, alpha=c.alpha,
                              out=o)
            for i in range(5):
                one(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = min(args.steps, 50)
            e0.record(stream)
            for i in range(n):
                one(i)
            e1.record(stream)
            torch.cuda.synchronize()
            line["context_cublas_fp32"] = {
                "value": flops_step / (e0.elapsed_time(e1) / n * 1e-3) / 1e12, "unit": UNIT,
                "what": "cuBLAS FP32 strided batch via torch.baddbmm, allow_tf32=False; context only"}
        finally:
            torch.backends.cuda.matmul.allow_tf32 = prev
    if not args.no_cpu_baseline:
        import oracle
        products, t = batched_oracle_sample(c, d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": products * si.flops(c.M, c.N, c.K) / t / 1e12, "unit": UNIT,
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"the first {products} of {c.batch} products ({c.M}x{c.N}x{c.K}) in {t:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    batched = {c.name: c for c in si.BATCHED_CASES}
    if args.config in batched:
        c = batched[args.config]
        if args.impl == "reference":
            run_reference_batched(args, c)
        else:
            run_ours_batched(args, c)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
