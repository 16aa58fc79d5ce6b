"""CPU tests: the oracle against its pins, and the input generators against the pages."""
import os

import numpy as np
import pytest

import oracle
import sgemm_inputs as si
from oracle_pins import ALL_PINS, GOLDEN


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(lib, pin):
    pin(lib)


def test_oracle_threads_reported(lib):
    assert oracle.num_threads() >= 1


# ---- input generators and workload counters -------------------------------------------------

def test_int_pattern_matches_c_semantics():
    want = np.loadtxt(os.path.join(GOLDEN, "int_pattern_4x5.txt"), dtype=np.float32)
    got = si.int_pattern(4, 5)
    assert np.array_equal(got, want)
    assert not np.any(np.signbit(got[got == 0]))      # zeros are +0.0, as an int->float cast gives


def test_uniform_range_and_reproducible():
    a = si.uniform_pm1(300, 200, seed=3, stream=1)
    b = si.uniform_pm1(300, 200, seed=3, stream=1)
    c = si.uniform_pm1(300, 200, seed=3, stream=2)
    assert a.dtype == np.float32 and np.array_equal(a, b) and not np.array_equal(a, c)
    assert a.min() >= -1.0 and a.max() < 1.0
    assert abs(float(a.mean())) < 0.02 and abs(float(a.var()) - 1.0 / 3.0) < 0.01


def test_normal_weights_scale():
    w = si.normal(4096, 64, seed=6, stream=2, std=1.0 / np.sqrt(1024))
    assert abs(float(w.std()) * np.sqrt(1024) - 1.0) < 0.01


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_flop_and_byte_counts_match_pages():
    for kind, M, N, K, beta, printed, rtol, *_ in _golden_rows("flop_counts.txt"):
        M, N, K, beta, printed, rtol = int(M), int(N), int(K), float(beta), float(printed), float(rtol)
        got = si.flops(M, N, K) if kind == "flops" else si.min_bytes(M, N, K, beta)
        assert abs(got - printed) <= rtol * printed, (kind, M, N, K, got, printed)


def test_rate_conversion_matches_page():
    for gflop, seconds, tflops in _golden_rows("rate_conversion.txt"):
        assert abs(float(gflop) * 1e9 / float(seconds) / 1e12 - float(tflops)) < 1e-9


def test_case_table_shapes():
    names = [c.name for c in si.CASES]
    assert len(set(names)) == len(names)
    h = si.case(si.HEADLINE)
    assert (h.M, h.N, h.K, h.transA, h.transB, h.alpha, h.beta) == (4096, 4096, 4096, "N", "N", 1.5, -0.5)
    r = si.case("ragged_TN")
    d = si.make_case(si.Case("tiny_ragged", 5, 6, 7, "T", "N", 1, 1, 5, "uniform", 7, "uniform"))
    assert d["A"].shape == (7, 5 + 7) and d["lda"] == 12 and np.all(np.isnan(d["A"][:, 5:]))
    assert d["B"].shape == (7, 6 + 7) and d["C"].shape == (5, 6 + 7)
    assert (r.M, r.N, r.K, r.pad) == (4097, 3001, 2053, 7)
