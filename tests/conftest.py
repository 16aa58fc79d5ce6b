"""pytest configuration: the ``gpu`` marker and the repository root on sys.path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libsgemm")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """The per-configuration parity figures of the GPU parity tests (when any ran)."""
    try:
        from gpu_util import PARITY_RECORDS
    except ImportError:
        return
    if not PARITY_RECORDS:
        return
    w = terminalreporter
    w.write_line("parity vs oracle: config / kernel / rows checked / worst err/bound / rel. Frobenius")
    for name, kernel, rows, worst, frob in PARITY_RECORDS:
        w.write_line(f"  {name:22s} {kernel:12s} {str(rows):>4s} {worst:9.3g} {frob:9.3g}")
