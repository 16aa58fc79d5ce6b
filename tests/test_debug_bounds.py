"""The bounds-checking build (libsgemm_debug.so: the kernels compiled with -DSGEMM_DEBUG_BOUNDS).

Every kernel checks each global-memory index (and the splitters their shared-
and tensor-memory offsets) against the buffer's extent before the access; a
violation is recorded and the access skipped, never trapped.  These GPU tests
run every kernel variant through the debug library on tiny, odd, ragged,
unaligned, split and batched shapes and require no recorded violation and the
oracle's results; the self-test shows that a violation is recorded (one check of
an index one past its limit, which is never dereferenced).  This stands in for
compute-sanitizer, which is closed on this machine.
"""
import ctypes

import numpy as np
import pytest

import oracle
import sgemm_inputs as si
import sgemm_row_major_gb300 as sg
from gpu_util import U, dyadic, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    from sgemm_row_major_gb300 import build
    build.build(debug=True)
    lib = sg.load_debug()
    assert lib.sgemm_debug_bounds_enabled() == 1
    return lib


def report(lib):
    site, off = ctypes.c_uint(0), ctypes.c_longlong(0)
    assert lib.sgemm_bounds_report(ctypes.byref(site), ctypes.byref(off)) == 0
    return site.value, off.value


def clean(lib):
    """Synchronise; no bounds violation may have been recorded."""
    st = lib.sgemm_sync_status(None)
    where = report(lib)
    assert st == 0 and where == (0, 0), f"status {st}, first violation (site, offset) {where}"


def test_selftest_records_a_violation(dbg):
    assert sg.load().sgemm_debug_bounds_enabled() == 0
    clean(dbg)
    assert dbg.sgemm_selftest_bounds(None) == 0
    assert dbg.sgemm_sync_status(None) == sg.STATUS["ERR_BOUNDS"]
    assert report(dbg) == (8, 64)
    assert report(dbg) == (0, 0)             # reading cleared it
    # the normal library has the checks compiled out: nothing is recorded
    lib = sg.load()
    assert lib.sgemm_selftest_bounds(None) == 0 and lib.sgemm_sync_status(None) == 0


def run(lib, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant="AUTO", split=0, offset=0, entry="sgemm"):
    torch = torch_cuda()
    dA = to_dev(np.concatenate([np.zeros(offset, np.float32), A.reshape(-1)]))
    dB = to_dev(np.concatenate([np.zeros(offset, np.float32), B.reshape(-1)]))
    dC = to_dev(C)
    lib.sgemm_set_variant_override(sg.VARIANTS[variant], split)
    try:
        args = (ta.encode(), tb.encode(), M, N, K, alpha, dA.data_ptr() + 4 * offset, lda, dB.data_ptr() + 4 * offset,
                ldb, beta, dC.data_ptr(), ldc, None)
        st = getattr(lib, entry)(*args)
    finally:
        lib.sgemm_set_variant_override(0, 0)
    assert st == 0, (entry, variant, st)
    clean(lib)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


SHAPES = [(1, 1, 1), (7, 5, 3), (33, 65, 16), (129, 130, 70), (300, 260, 1000), (513, 257, 95), (64, 700, 2049)]
VARIANTS = [("AUTO", 0), ("GENERIC", 0), ("GENERIC", 3), ("TMA_128x128", 0), ("TMA_128x128", 4), ("TMA_64x256", 0),
            ("TC_TF32X3", 0), ("TC_TF32X3", 3), ("TC_PAIR", 0), ("TC_PAIR", 3), ("TC_PRESPLIT", 0),
            ("TC_PRESPLIT", 3), ("TC_SKINNY", 0), ("TC_SKINNY", 3)]


@pytest.mark.parametrize("variant,split", VARIANTS, ids=[f"{v}-{s}" for v, s in VARIANTS])
@pytest.mark.parametrize("ops", ["NN", "NT", "TN", "TT"])
def test_variants_clean_and_exact(dbg, variant, split, ops):
    """Dyadic inputs (exact on every path), padded rows with NaN, alpha and beta."""
    ta, tb = ops
    rng = np.random.default_rng(sum(map(ord, f"{variant}{split}{ops}")))
    for M, N, K in SHAPES:
        ar, ac = si.stored_shape(ta, M, K)
        br, bc = si.stored_shape(tb, K, N)
        lda, ldb = (ac + 3) // 4 * 4 + 4, (bc + 3) // 4 * 4 + 8  # multiples of 4: TMA can load them
        A = si.embed_padded(dyadic(rng, ar, ac), lda)
        B = si.embed_padded(dyadic(rng, br, bc), ldb)
        C = dyadic(rng, M, N)
        got = run(dbg, ta, tb, M, N, K, 1.5, A, lda, B, ldb, -0.5, C, N, variant, split)
        ref = oracle.sgemm(ta, tb, A[:, :ac], B[:, :bc], C, 1.5, -0.5, M=M, N=N, K=K)
        assert np.array_equal(got, ref), (variant, split, ops, M, N, K)


@pytest.mark.parametrize("ops", ["NN", "TT"])
def test_unaligned_and_tf32_clean(dbg, ops):
    """Operands one float off alignment with odd leading dimensions (generic kernel and the
    split-operand kernel's any-alignment split pass), and the TF32- and BF16-input entry points."""
    ta, tb = ops
    rng = np.random.default_rng(5)
    for M, N, K in [(203, 157, 301), (700, 650, 1203)]:
        ar, ac = si.stored_shape(ta, M, K)
        br, bc = si.stored_shape(tb, K, N)
        A = si.embed_padded(dyadic(rng, ar, ac), ac + 3)
        B = si.embed_padded(dyadic(rng, br, bc), bc + 1)
        C = dyadic(rng, M, N)
        got = run(dbg, ta, tb, M, N, K, 1.0, A, ac + 3, B, bc + 1, 1.0, C, N, offset=1)
        assert np.array_equal(got, oracle.sgemm(ta, tb, A[:, :ac], B[:, :bc], C, 1.0, 1.0, M=M, N=N, K=K))
        got = run(dbg, ta, tb, M, N, K, 1.0, A, ac + 3, B, bc + 1, 1.0, C, N, offset=1, entry="sgemm_tf32")
        assert np.array_equal(got, oracle.sgemm_tf32(ta, tb, A[:, :ac], B[:, :bc], C, 1.0, 1.0, M=M, N=N, K=K))
        got = run(dbg, ta, tb, M, N, K, 1.0, A, ac + 3, B, bc + 1, 1.0, C, N, offset=1, entry="sgemm_bf16")
        assert np.array_equal(got, oracle.sgemm_bf16(ta, tb, A[:, :ac], B[:, :bc], C, 1.0, 1.0, M=M, N=N, K=K))


def test_noalloc_and_scale_clean(dbg):
    rng = np.random.default_rng(6)
    M, N, K = 300, 520, 1000
    A, B, C = dyadic(rng, M, K), dyadic(rng, K, N), dyadic(rng, M, N)
    got = run(dbg, "N", "N", M, N, K, 2.0, A, K, B, N, 0.5, C, N, entry="sgemm_noalloc")
    assert np.array_equal(got, oracle.sgemm("N", "N", A, B, C, 2.0, 0.5))
    got = run(dbg, "N", "N", M, N, 0, 2.0, A, K, B, N, 0.5, C, N)        # K = 0: C = beta C
    assert np.array_equal(got, (0.5 * C.astype(np.float64)).astype(np.float32))


@pytest.mark.parametrize("variant,M,N,K,batch", [("AUTO", 36, 20, 300, 305), ("TC_GROUPED", 20, 28, 100, 7),
                                                 ("SMALL", 36, 20, 100, 50), ("AUTO", 300, 270, 601, 6),
                                                 ("TC_PRESPLIT", 200, 300, 96, 5), ("GENERIC", 97, 70, 131, 4)])
def test_batched_clean(dbg, variant, M, N, K, batch):
    """Strided batches with NaN padding and gaps (odd strides for the generic kernel and the
    split-operand kernel's split pass)."""
    torch = torch_cuda()
    align = 1 if variant in ("GENERIC",) or (variant == "AUTO" and M == 300) else 4
    d = si.make_batched(batch, M, N, K, "N", "N", seed=7, pad=1 if align == 1 else 4, gap=3, align=align)
    rng = np.random.default_rng(8)
    for name in "ABC":
        X = d["stacks"][name]
        d["stacks"][name] = (rng.integers(-64, 64, size=X.shape) / 64).astype(np.float32)
        d[name] = si.embed_batched(d["stacks"][name], d["ld" + name.lower()], d["stride" + name])
    dA, dB, dC = to_dev(d["A"]), to_dev(d["B"]), to_dev(d["C"])
    dbg.sgemm_set_variant_override(sg.VARIANTS[variant], 0)
    try:
        st = dbg.sgemm_strided_batched(b"N", b"N", M, N, K, 1.5, dA.data_ptr(), d["lda"], dB.data_ptr(), d["ldb"],
                                       -0.5, dC.data_ptr(), d["ldc"], d["strideA"], d["strideB"], d["strideC"],
                                       batch, None)
    finally:
        dbg.sgemm_set_variant_override(0, 0)
    assert st == 0
    clean(dbg)
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    ref, _ = oracle.sgemm_strided_batched("N", "N", M, N, K, 1.5, d["A"], d["lda"], d["strideA"], d["B"], d["ldb"],
                                          d["strideB"], -0.5, d["C"], d["ldc"], d["strideC"], batch, want_bound=True)
    assert np.array_equal(got, ref, equal_nan=True)
