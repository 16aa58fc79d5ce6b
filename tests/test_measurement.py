"""GPU test of the measurement aid: per-SM clock snapshots around a stretch of
GEMM work give every SM's average clock over it (cycle-counter delta over
global-timer delta), a plausible SM frequency."""
import pytest

import bench
import sgemm_row_major_gb300 as sg
from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu


def test_clock_snapshot_gives_sm_clock():
    torch = torch_cuda()
    n = 2048
    A = torch.rand(n, n, device="cuda")
    B = torch.rand(n, n, device="cuda")
    C = torch.empty(n, n, device="cuda")
    before = torch.zeros(2 * 1024, dtype=torch.int64, device="cuda")
    after = torch.zeros(2 * 1024, dtype=torch.int64, device="cuda")
    sg.sgemm("N", "N", n, n, n, 1.0, A, n, B, n, 0.0, C, n)
    sg.sgemm_clock_snapshot(before)
    for _ in range(20):
        sg.sgemm("N", "N", n, n, n, 1.0, A, n, B, n, 0.0, C, n)
    sg.sgemm_clock_snapshot(after)
    torch.cuda.synchronize()
    assert sg.sgemm_sync_status() == 0
    mhz, sms = bench.snapshot_mhz(before, after)
    assert sms >= torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert 300.0 < mhz < 3000.0, mhz
    with pytest.raises(sg.SgemmError):
        sg.sgemm_clock_snapshot(torch.zeros(1, dtype=torch.int64, device="cuda"))  # fewer than one slot
