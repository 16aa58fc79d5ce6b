"""The committed ncu summaries that bench.py reads DRAM traffic from: each
exists, names the kernel digest and per-launch traffic it was captured with,
and gives the commands that made it (never a capture that locks clocks)."""
import os
import re

import bench


def test_every_profile_entry_parses():
    assert bench.PROFILES
    for (variant, workload), path in bench.PROFILES.items():
        assert os.path.exists(path), path
        text = open(path).read()
        assert re.search(r"^kernel_digest: [0-9a-f]{16}$", text, re.M), path
        t = re.search(r"^traffic_bytes_per_launch: ([0-9]+)$", text, re.M)
        assert t and int(t.group(1)) > 0, path
        cmds = [line for line in text.splitlines() if line.strip().startswith("ncu ")]
        assert cmds and all("--clock-control none" in c for c in cmds), path
        assert workload in text or workload == "square4096", (path, workload)


def test_traffic_only_for_the_matching_digest():
    (variant, workload), path = next(iter(bench.PROFILES.items()))
    digest = re.search(r"^kernel_digest: ([0-9a-f]+)$", open(path).read(), re.M).group(1)
    assert bench.traffic_from_profile(variant, workload, digest) > 0
    assert bench.traffic_from_profile(variant, workload, "0" * 16) is None
    assert bench.traffic_from_profile(variant, "no_such_workload", digest) is None
