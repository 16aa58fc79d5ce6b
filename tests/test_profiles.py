"""The committed ncu capture record bench.py reads DRAM traffic from
(profiles/traffic.json): every entry names its kernel variant, workload,
kernel digest and per-launch traffic, and points at an existing summary that
gives the commands that made it (never a capture that locks clocks)."""
import json
import os

import bench


def entries():
    return json.load(open(bench.TRAFFIC_FILE))["entries"]


def test_every_traffic_entry_is_complete():
    es = entries()
    assert es
    seen = set()
    for e in es:
        key = (e["variant"], e["workload"])
        assert key not in seen, key
        seen.add(key)
        assert len(e["kernel_digest"]) == 16 and int(e["kernel_digest"], 16) >= 0
        assert int(e["traffic_bytes_per_launch"]) > 0
        path = os.path.join(bench.ROOT, e["summary"])
        assert os.path.exists(path), path
        text = open(path).read()
        cmds = [line for line in text.splitlines() if line.strip().startswith("ncu ")]
        assert cmds and all("--clock-control none" in c for c in cmds), path


def test_traffic_only_for_the_matching_digest():
    e = entries()[0]
    assert bench.traffic_from_profile(e["variant"], e["workload"], e["kernel_digest"]) == e["traffic_bytes_per_launch"]
    assert bench.traffic_from_profile(e["variant"], e["workload"], "0" * 16) is None
    assert bench.traffic_from_profile(e["variant"], "no_such_workload", e["kernel_digest"]) is None


def test_snapshot_clock_from_counter_deltas():
    import torch
    b = torch.zeros(8, dtype=torch.int64)
    a = torch.zeros(8, dtype=torch.int64)
    # SM 0: 2.0e6 cycles in 1.0e6 ns (2000 MHz); SM 1: 1.9e6 in 1.0e6 (1900 MHz); SMs 2, 3 never ran
    b[0], b[1], a[0], a[1] = 100, 5_000_000, 2_000_100, 6_000_000
    b[2], b[3], a[2], a[3] = 7, 5_000_000, 1_900_007, 6_000_000
    mhz, n = bench.snapshot_mhz(b, a)
    assert n == 2 and abs(mhz - 1950.0) < 1e-6


def test_hbm_roof_chosen_when_bytes_bind():
    peaks = {"hbm_gbs": 6781.4, "bf16_tflops": 1910.0}
    # skinny 64 x 4096 x 16384: 273.7 MB at HBM (40 us) outlast 8.6 GFLOP at the 3xTF32 peak (28 us)
    roof = bench.tensor_roofline(100.0, peaks, None, 0.08)
    bench.hbm_bound_roofline(roof, 273.7e6, 8.59e9, 0.08, peaks)
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["tensor"]["unit"] == "TFLOP/s"
    assert abs(roof["achieved"] - 273.7e6 / 0.08e-3 / 1e9) < 1e-6
    # 4096^3: tensor-bound
    roof = bench.tensor_roofline(270.0, peaks, None, 0.5)
    bench.hbm_bound_roofline(roof, 268.4e6, 137.4e9, 0.5, peaks)
    assert roof["bound"] == "tensor"


def test_l2_hot_block():
    """Configs whose input set fits in L2 carry an L2-hot figure beside the flushed one; larger
    ones say why they have none."""
    assert bench.l2_hot_block(None, None, 1e9)["value"] is None
    hot = bench.l2_hot_block(lambda: None, 0.01, 2.147e9)  # 10 us per 1024^3 step
    assert abs(hot["value"] - 214.7) < 1e-9 and hot["unit"] == "TFLOPS" and hot["ms_per_step"] == 0.01


def test_reduced_precision_entries():
    """bench.py --entry tf32 / bf16: the library, plan and oracle functions it names exist, the
    roofline takes the measured bf16 peak (BF16 inputs) or that peak x 1.1/2.25 (TF32 inputs),
    and the config names the entry point only when it is not sgemm()."""
    import oracle
    import sgemm_row_major_gb300 as sg
    for e, (lib_fn, plan_fn, oracle_fn, dtype) in bench.ENTRIES.items():
        assert callable(getattr(sg, lib_fn)) and callable(getattr(sg, plan_fn)) and callable(getattr(oracle, oracle_fn))
        assert dtype
    peaks = {"bf16_tflops": 1910.0}
    bf = bench.reduced_roofline(955.0, peaks, "TC_BF16", 0.144, None)
    assert bf["bound"] == "tensor" and bf["peak"] == 1910.0 and abs(bf["frac"] - 0.5) < 1e-12
    tf = bench.reduced_roofline(467.0, peaks, "TC_TF32", 0.294, None)
    assert abs(tf["peak"] - 1910.0 * 1.1 / 2.25) < 1e-9 and abs(tf["frac"] - 467.0 / tf["peak"]) < 1e-12
    import sgemm_inputs as si
    c = si.case("square4096")
    assert "entry" not in bench.config_block(c, 1)
    assert bench.config_block(c, 1, "sgemm_bf16")["entry"] == "sgemm_bf16"
