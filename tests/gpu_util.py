"""Helpers for the GPU tests: device copies, oracle on sampled rows, error checks."""
from __future__ import annotations

import numpy as np

import oracle
import sgemm_inputs as si

U = 2.0 ** -24           # unit roundoff of float32
FROB_LIMIT = 1e-6        # relative Frobenius error limit on random inputs

# (config, kernel, rows checked, worst err/bound, relative Frobenius error) of the parity tests,
# printed at the end of the run by conftest.py
PARITY_RECORDS: list = []


def record_parity(name, kernel, rows, worst, frob):
    PARITY_RECORDS.append((name, kernel, rows, worst, frob))


def torch_cuda():
    import torch
    return torch


def to_dev(x: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def gpu_sgemm(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant=None, split=0, stream=None):
    """Run libsgemm on numpy operands (stored, possibly padded); returns the full C buffer."""
    import sgemm_row_major_gb300 as sg
    torch = torch_cuda()
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    if variant is not None or split:
        sg.sgemm_set_variant_override(variant or "AUTO", split)
    try:
        sg.sgemm(ta, tb, M, N, K, alpha, dA, lda, dB, ldb, beta, dC, ldc, stream=stream)
    finally:
        if variant is not None or split:
            sg.sgemm_set_variant_override("AUTO", 0)
    assert sg.sgemm_sync_status(stream) == 0
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def sample_rows(M: int, n: int, seed: int, tile: int = 128) -> np.ndarray:
    rng = np.random.default_rng(seed)
    fixed = {0, 1, M - 1, M - 2, min(tile - 1, M - 1), min(tile, M - 1), M // 2}
    extra = rng.choice(M, size=min(n, M), replace=False)
    return np.array(sorted(fixed | set(int(r) for r in extra)), dtype=np.int64)


def oracle_rows(case: si.Case, d: dict, rows: np.ndarray | None):
    """Oracle C (and S) for the given rows of C (all rows when None)."""
    M, N, K = case.M, case.N, case.K
    A = d["A"][:, :(M if case.transA == "T" else K)]
    B = d["B"][:, :(K if case.transB == "T" else N)]
    C = d["C"][:, :N]
    if rows is not None:
        A = np.ascontiguousarray(A[:, rows] if case.transA == "T" else A[rows, :])
        C = np.ascontiguousarray(C[rows, :])
        M = len(rows)
    return oracle.sgemm(case.transA, case.transB, A, B, C, case.alpha, case.beta, M=M, N=N, K=K,
                        want_bound=True)


def check_bound(got: np.ndarray, ref: np.ndarray, S: np.ndarray, K: int, what: str = ""):
    """Per element |got - ref| <= (K + 2) u S, and the relative Frobenius error <= 1e-6."""
    got64, ref64 = got.astype(np.float64), ref.astype(np.float64)
    assert np.all(np.isfinite(got64)), f"{what}: non-finite output"
    err = np.abs(got64 - ref64)
    bound = (K + 2) * U * S
    worst = float(np.max(err / np.maximum(bound, 1e-300)))
    assert np.all(err <= bound), f"{what}: per-element bound violated, worst err/bound = {worst:.3g}"
    frob = float(np.linalg.norm(got64 - ref64) / max(np.linalg.norm(ref64), 1e-300))
    assert frob <= FROB_LIMIT, f"{what}: relative Frobenius error {frob:.3g} > {FROB_LIMIT}"
    return worst, frob


def check_exact(got: np.ndarray, ref: np.ndarray, what: str = ""):
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{what}: {len(bad)} elements differ, first at {tuple(bad[0])}: {got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}"


def dyadic(rng, rows, cols, bits=6):
    """Multiples of 2^-bits in [-1, 1): short significands make every partial sum exact in float32."""
    scale = 2 ** bits
    return (rng.integers(-scale, scale, size=(rows, cols)) / scale).astype(np.float32)
