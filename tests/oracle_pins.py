"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each ``pin_*`` takes an oracle ctypes library (``oracle.load_library``) and
raises AssertionError when the oracle disagrees with:
  * a worked example (tests/golden/hand_2x2.txt),
  * an independent float64 ``np.einsum`` on tiny shapes with dyadic inputs,
    where every partial sum is exact, so the result is unique,
  * an int64 matmul on the pages' integer fill (exact in float32 and double),
  * closed forms and invariants (K=1 correctly rounded product, alpha=0,
    beta=0 with NaN in C, identity, (AB)^T = B^T A^T, op='T' of a transposed
    copy, exact power-of-two scaling of alpha, padding never read),
  * a float64 BLAS matmul at a medium size within the final rounding,
  * the bound magnitude S = |alpha| |A|@|B| + |beta C|,
  * exact rational arithmetic, correctly rounded once, on values at the top of
    the float32 range, and the IEEE 754 rules for Inf and NaN operands,
  * for the TF32-input GEMM: hand-worked roundings (tests/golden/tf32_round.txt),
    a bit-level characterization of the rounding over all exponents, and a
    float64 einsum of independently rounded tiny inputs; the same three for the
    BF16-input GEMM (tests/golden/bf16_round.txt, ties to even).
The same pins run against deliberately broken copies of the oracle in
test_oracle_mutations.py, which shows that each plausible mistake fails one.
"""
from __future__ import annotations

import itertools
import os
from fractions import Fraction

import numpy as np

import oracle
import sgemm_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

OPS = [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")]


def _op(X: np.ndarray, t: str) -> np.ndarray:
    return X.T if t == "T" else X


def _stored(rng, op, rows, cols, dyadic_bits=None):
    shp = si.stored_shape(op, rows, cols)
    if dyadic_bits is None:
        return (2.0 * rng.random(shp) - 1.0).astype(np.float32)
    scale = 2 ** dyadic_bits
    return (rng.integers(-scale, scale, size=shp) / scale).astype(np.float32)


def read_golden_matrix_file(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = np.array([float(v) for v in vals], dtype=np.float32)
    return rows


def pin_hand_2x2(lib):
    g = read_golden_matrix_file("hand_2x2.txt")
    A, B, C = (g[k].reshape(2, 2) for k in "ABC")
    out = oracle.sgemm("N", "N", A, B, lib=lib)
    assert np.array_equal(out, C), out


def pin_bruteforce_tiny(lib):
    """All 4 ops, M,N,K in {1,2,3,5,7}, alpha/beta in {0,1,-0.5,2}: equal to float64 einsum.

    Inputs are multiples of 2^-6 in [-1, 1), so products have <= 14 significant
    bits and every partial sum is exact in double: any summation order gives
    the same double, and one rounding to float32 gives a unique answer.
    """
    rng = np.random.default_rng(1234)
    sizes = [1, 2, 3, 5, 7]
    scalars = [0.0, 1.0, -0.5, 2.0]
    for (ta, tb), M, N, K in itertools.product(OPS, sizes, sizes, sizes):
        A = _stored(rng, ta, M, K, dyadic_bits=6)
        B = _stored(rng, tb, K, N, dyadic_bits=6)
        C = _stored(rng, "N", M, N, dyadic_bits=6)
        alpha, beta = scalars[rng.integers(4)], scalars[rng.integers(4)]
        ref = (alpha * np.einsum("ik,kj->ij", _op(A, ta).astype(np.float64), _op(B, tb).astype(np.float64))
               + beta * C.astype(np.float64)).astype(np.float32)
        out = oracle.sgemm(ta, tb, A, B, C, alpha, beta, lib=lib)
        assert np.array_equal(out, ref), (ta, tb, M, N, K, alpha, beta)


def pin_integer_pattern(lib, M=1000, N=1300, K=700, ops=OPS):
    """The pages' (j-i)%3 fill on both stored operands: equal to an int64 matmul."""
    for ta, tb in ops:
        A = si.int_pattern(*si.stored_shape(ta, M, K))
        B = si.int_pattern(*si.stored_shape(tb, K, N))
        ref = _op(A, ta).astype(np.int64) @ _op(B, tb).astype(np.int64)
        assert np.abs(ref).max() < 2 ** 24
        out = oracle.sgemm(ta, tb, A, B, lib=lib)
        assert np.array_equal(out, ref.astype(np.float32)), (ta, tb)


def pin_integer_alpha_beta(lib, M=37, N=41, K=53):
    """Integer fill with alpha=1.5, beta=-0.5 and integer C: exact in float32."""
    rng = np.random.default_rng(7)
    for ta, tb in OPS:
        A = si.int_pattern(*si.stored_shape(ta, M, K))
        B = si.int_pattern(*si.stored_shape(tb, K, N))
        C = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
        ref = 1.5 * (_op(A, ta).astype(np.int64) @ _op(B, tb).astype(np.int64)) - 0.5 * C.astype(np.float64)
        out = oracle.sgemm(ta, tb, A, B, C, 1.5, -0.5, lib=lib)
        assert np.array_equal(out, ref.astype(np.float32)), (ta, tb)


def pin_k1_exact(lib):
    """K=1, alpha=1, beta=0: each element is one correctly rounded float32 product."""
    rng = np.random.default_rng(5)
    for ta, tb in OPS:
        A = _stored(rng, ta, 23, 1)
        B = _stored(rng, tb, 1, 29)
        ref = _op(A, ta).astype(np.float32) * _op(B, tb).astype(np.float32)  # float32 IEEE multiply
        out = oracle.sgemm(ta, tb, A, B, lib=lib)
        assert np.array_equal(out, ref), (ta, tb)


def pin_alpha_zero(lib):
    """alpha = 0: C = fl32(beta*C) and A, B are not read (NaN operands do not leak)."""
    rng = np.random.default_rng(6)
    A = np.full((9, 11), np.nan, np.float32)
    B = np.full((11, 13), np.nan, np.float32)
    C = _stored(rng, "N", 9, 13)
    for beta in (0.0, 1.0, -0.5, 3.0):
        out = oracle.sgemm("N", "N", A, B, C, 0.0, beta, lib=lib)
        assert np.array_equal(out, (np.float64(beta) * C.astype(np.float64)).astype(np.float32)), beta


def pin_k_zero(lib):
    """K = 0: C = fl32(beta*C)."""
    rng = np.random.default_rng(16)
    C = _stored(rng, "N", 5, 6)
    A = np.zeros((5, 0), np.float32)
    B = np.zeros((0, 6), np.float32)
    out = oracle.sgemm("N", "N", A, B, C, 2.0, -0.5, M=5, N=6, K=0, lib=lib)
    assert np.array_equal(out, (-0.5 * C.astype(np.float64)).astype(np.float32))


def pin_beta_zero_nan_c(lib):
    """beta = 0: C is not read, so a NaN-filled C gives the same result as a zero C."""
    rng = np.random.default_rng(8)
    for ta, tb in OPS:
        A = _stored(rng, ta, 17, 19)
        B = _stored(rng, tb, 19, 15)
        Cnan = np.full((17, 15), np.nan, np.float32)
        out = oracle.sgemm(ta, tb, A, B, Cnan, 1.25, 0.0, lib=lib)
        ref = oracle.sgemm(ta, tb, A, B, None, 1.25, 0.0, lib=lib)
        assert np.all(np.isfinite(out)) and np.array_equal(out, ref), (ta, tb)


def pin_identity(lib):
    """op(A) = I: C = fl32(alpha*B + beta*C)."""
    rng = np.random.default_rng(9)
    n = 31
    eye = np.eye(n, dtype=np.float32)
    for ta in "NT":
        B = _stored(rng, "N", n, 24)
        C = _stored(rng, "N", n, 24)
        out = oracle.sgemm(ta, "N", eye, B, C, 0.75, -1.5, lib=lib)
        ref = (0.75 * B.astype(np.float64) - 1.5 * C.astype(np.float64)).astype(np.float32)
        assert np.array_equal(out, ref), ta


def pin_transpose_identity(lib):
    """(AB)^T = B^T A^T: sgemm('T','T', N, M, K, B, A) equals the transpose of sgemm('N','N')."""
    rng = np.random.default_rng(10)
    A = _stored(rng, "N", 33, 47)
    B = _stored(rng, "N", 47, 29)
    C = oracle.sgemm("N", "N", A, B, lib=lib)
    Ct = oracle.sgemm("T", "T", B, A, lib=lib)          # stored B is K x N -> op(B^T) is N x K
    assert Ct.shape == (29, 33)
    assert np.array_equal(Ct, C.T)                       # same products, same k order


def pin_transposed_copy(lib):
    """op='T' on an explicitly transposed copy equals op='N' on the original."""
    rng = np.random.default_rng(11)
    A = _stored(rng, "N", 21, 34)
    B = _stored(rng, "N", 34, 18)
    C = _stored(rng, "N", 21, 18)
    ref = oracle.sgemm("N", "N", A, B, C, 1.5, -0.5, lib=lib)
    At = np.ascontiguousarray(A.T)
    Bt = np.ascontiguousarray(B.T)
    for ta, tb, AA, BB in (("T", "N", At, B), ("N", "T", A, Bt), ("T", "T", At, Bt)):
        out = oracle.sgemm(ta, tb, AA, BB, C, 1.5, -0.5, lib=lib)
        assert np.array_equal(out, ref), (ta, tb)


def pin_alpha_pow2(lib):
    """alpha * 2^e scales C exactly when beta = 0 (no overflow/underflow)."""
    rng = np.random.default_rng(12)
    A = _stored(rng, "N", 19, 26)
    B = _stored(rng, "N", 26, 23)
    base = oracle.sgemm("N", "N", A, B, None, 0.75, 0.0, lib=lib)
    for e in (-3, 1, 5):
        out = oracle.sgemm("N", "N", A, B, None, 0.75 * 2.0 ** e, 0.0, lib=lib)
        assert np.array_equal(out, (base.astype(np.float64) * 2.0 ** e).astype(np.float32)), e


def pin_padding_not_read(lib):
    """Row strides larger than the logical width: NaN padding never reaches C."""
    rng = np.random.default_rng(13)
    for ta, tb in OPS:
        A = _stored(rng, ta, 14, 22)
        B = _stored(rng, tb, 22, 17)
        C = _stored(rng, "N", 14, 17)
        ref = oracle.sgemm(ta, tb, A, B, C, 1.0, 1.0, lib=lib)
        Ap = si.embed_padded(A, A.shape[1] + 7)
        Bp = si.embed_padded(B, B.shape[1] + 5)
        out = oracle.sgemm(ta, tb, Ap[:, :A.shape[1]], Bp[:, :B.shape[1]], C, 1.0, 1.0, lib=lib)
        assert np.array_equal(out, ref), (ta, tb)
        # and the raw interface with a padded C: padding of C is left untouched
        Cp = si.embed_padded(C, 17 + 3)
        flatC = Cp.reshape(-1).copy()
        st = oracle.sgemm_raw(ta, tb, 14, 17, 22, 1.0, Ap.reshape(-1), Ap.shape[1], Bp.reshape(-1), Bp.shape[1],
                              1.0, flatC, 20, lib=lib)
        assert st == 0
        got = flatC.reshape(14, 20)
        assert np.array_equal(got[:, :17], ref) and np.all(np.isnan(got[:, 17:])), (ta, tb)


def pin_random_vs_float64_matmul(lib, M=150, N=170, K=700):
    """Random uniform inputs: within the final float32 rounding of a float64 BLAS matmul."""
    rng = np.random.default_rng(14)
    for ta, tb in OPS:
        A = _stored(rng, ta, M, K)
        B = _stored(rng, tb, K, N)
        C = _stored(rng, "N", M, N)
        ref = 1.5 * (_op(A, ta).astype(np.float64) @ _op(B, tb).astype(np.float64)) - 0.5 * C.astype(np.float64)
        out = oracle.sgemm(ta, tb, A, B, C, 1.5, -0.5, lib=lib).astype(np.float64)
        absref = 1.5 * (np.abs(_op(A, ta)).astype(np.float64) @ np.abs(_op(B, tb)).astype(np.float64)) \
            + 0.5 * np.abs(C.astype(np.float64))
        # one float32 rounding (2^-24 |ref|) plus double-precision summation noise
        err = np.abs(out - ref)
        assert np.all(err <= 2.0 ** -24 * np.abs(ref) + 1e-12 * absref), (ta, tb, err.max())


def pin_bound_magnitude(lib):
    """S_ij = |alpha| sum_k |a_ik b_kj| + |beta c_ij|, against |A| @ |B| in float64."""
    rng = np.random.default_rng(15)
    for ta, tb in OPS:
        A = _stored(rng, ta, 12, 40)
        B = _stored(rng, tb, 40, 10)
        C = _stored(rng, "N", 12, 10)
        _, S = oracle.sgemm(ta, tb, A, B, C, -2.0, -0.5, want_bound=True, lib=lib)
        ref = 2.0 * (np.abs(_op(A, ta)).astype(np.float64) @ np.abs(_op(B, tb)).astype(np.float64)) \
            + 0.5 * np.abs(C.astype(np.float64))
        assert np.allclose(S, ref, rtol=1e-13, atol=0), (ta, tb)


def pin_argument_errors(lib):
    """Invalid arguments are rejected with -(argument index), BLAS style."""
    A = np.zeros(16, np.float32)
    cases = [
        (("X", "N", 2, 2, 2, 2, 2, 2), -1),
        (("N", "Q", 2, 2, 2, 2, 2, 2), -2),
        (("N", "N", -1, 2, 2, 2, 2, 2), -3),
        (("N", "N", 2, -1, 2, 2, 2, 2), -4),
        (("N", "N", 2, 2, -1, 2, 2, 2), -5),
        (("N", "N", 2, 2, 3, 2, 2, 2), -8),     # lda < K
        (("T", "N", 3, 2, 2, 2, 2, 2), -8),     # lda < M for 'T'
        (("N", "N", 2, 3, 2, 2, 2, 3), -10),    # ldb < N
        (("N", "T", 2, 2, 3, 3, 2, 2), -10),    # ldb < K for 'T'
        (("N", "N", 2, 3, 2, 2, 3, 2), -13),    # ldc < N
    ]
    for (ta, tb, M, N, K, lda, ldb, ldc), want in cases:
        st = oracle.sgemm_raw(ta, tb, M, N, K, 1.0, A, lda, A, ldb, 0.0, A.copy(), ldc, lib=lib)
        assert st == want, ((ta, tb, M, N, K, lda, ldb, ldc), st, want)


def pin_conjugate_is_transpose(lib):
    """'C' (conjugate transpose) on real data is 'T'; lower-case letters are accepted."""
    rng = np.random.default_rng(17)
    A = _stored(rng, "T", 9, 12)
    B = _stored(rng, "T", 12, 8)
    ref = oracle.sgemm("T", "T", A, B, lib=lib)
    for ta, tb in (("C", "C"), ("c", "t"), ("t", "C")):
        assert np.array_equal(oracle.sgemm(ta, tb, A, B, lib=lib), ref), (ta, tb)
    An = _stored(rng, "N", 9, 12)
    assert np.array_equal(oracle.sgemm("n", "t", An, B, lib=lib), oracle.sgemm("N", "T", An, B, lib=lib))


def _dyadic_stack(rng, n, rows, cols, bits=6):
    scale = 2 ** bits
    return (rng.integers(-scale, scale, size=(n, rows, cols)) / scale).astype(np.float32)


def pin_batched_dyadic(lib):
    """Strided batch: each product equals a float64 einsum over the stacked
    dyadic operands (exact), for every op, with odd strides, NaN gaps between
    matrices (never read, never written) and one shared operand (stride 0);
    S of product b is that product's |alpha| |A_b|@|B_b| + |beta C_b|."""
    rng = np.random.default_rng(18)
    batch, M, N, K = 4, 5, 6, 7
    alpha, beta = -1.5, 0.5
    for (ta, tb), shared in itertools.product(OPS, ("", "A", "B")):
        a_shape, b_shape = si.stored_shape(ta, M, K), si.stored_shape(tb, K, N)
        A = _dyadic_stack(rng, 1 if shared == "A" else batch, *a_shape)
        B = _dyadic_stack(rng, 1 if shared == "B" else batch, *b_shape)
        C = _dyadic_stack(rng, batch, M, N)
        lda, ldb, ldc = a_shape[1] + 1, b_shape[1] + 2, N + 3
        sa = 0 if shared == "A" else a_shape[0] * lda + 5
        sb = 0 if shared == "B" else b_shape[0] * ldb + 3
        sc = M * ldc + 1
        Af, Bf, Cf = si.embed_batched(A, lda, sa), si.embed_batched(B, ldb, sb), si.embed_batched(C, ldc, sc)
        out, S = oracle.sgemm_strided_batched(ta, tb, M, N, K, alpha, Af, lda, sa, Bf, ldb, sb, beta, Cf, ldc, sc,
                                              batch, want_bound=True, lib=lib)
        opA = np.stack([_op(A[0 if shared == "A" else b], ta) for b in range(batch)]).astype(np.float64)
        opB = np.stack([_op(B[0 if shared == "B" else b], tb) for b in range(batch)]).astype(np.float64)
        ref = (alpha * np.einsum("bik,bkj->bij", opA, opB) + beta * C.astype(np.float64)).astype(np.float32)
        want = si.embed_batched(ref, ldc, sc)
        assert np.array_equal(out, want, equal_nan=True), (ta, tb, shared)
        sref = abs(alpha) * np.einsum("bik,bkj->bij", np.abs(opA), np.abs(opB)) + abs(beta) * np.abs(C)
        assert np.array_equal(S, sref), (ta, tb, shared)


def pin_batched_edges(lib):
    """batch_count 0 leaves C untouched; one product equals the plain SGEMM;
    negative strides or counts are rejected."""
    rng = np.random.default_rng(19)
    A = _dyadic_stack(rng, 1, 4, 3)
    B = _dyadic_stack(rng, 1, 3, 5)
    C = _dyadic_stack(rng, 1, 4, 5)
    Af, Bf, Cf = A.ravel(), B.ravel(), C.ravel()
    out = oracle.sgemm_strided_batched("N", "N", 4, 5, 3, 1.0, Af, 3, 12, Bf, 5, 15, 2.0, Cf, 5, 20, 0, lib=lib)
    assert np.array_equal(out, Cf)
    one = oracle.sgemm_strided_batched("N", "N", 4, 5, 3, 1.0, Af, 3, 12, Bf, 5, 15, 2.0, Cf, 5, 20, 1, lib=lib)
    ref = (A[0].astype(np.float64) @ B[0].astype(np.float64) + 2.0 * C[0]).astype(np.float32)
    assert np.array_equal(one.reshape(4, 5), ref)
    for bad in ((-1, 15, 20, 2), (12, -1, 20, 2), (12, 15, -1, 2), (12, 15, 20, -1)):
        try:
            oracle.sgemm_strided_batched("N", "N", 4, 5, 3, 1.0, Af, 3, bad[0], Bf, 5, bad[1], 2.0, Cf, 5, bad[2],
                                         bad[3], lib=lib)
        except oracle.OracleError:
            continue
        raise AssertionError(f"accepted {bad}")


def _round_f32(x: Fraction) -> np.float32:
    """x rounded to the nearest float32 (ties to an even significand), from exact arithmetic."""
    c = np.float32(float(x))
    best = None
    for y in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        if not np.isfinite(y):
            continue
        d = abs(Fraction(float(y)) - x)
        key = (d, int(np.float32(y).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, y)
    return np.float32(best[1])


def pin_large_finite_exact(lib):
    """Values near FLT_MAX (2^128 (1 - 2^-13), FLT_MAX) times small ones, with alpha and beta:
    the oracle equals the exact rational result rounded to float32 once."""
    rng = np.random.default_rng(17)
    big = [np.float32((2 - 2.0 ** -12) * 2.0 ** 127), np.finfo(np.float32).max, np.float32(-(2 - 2.0 ** -11) * 2.0 ** 127)]
    for trial in range(40):
        M, N, K = (int(v) for v in rng.integers(1, 5, size=3))
        a = (rng.integers(-64, 64, size=(M, K)) / 64.0).astype(np.float32)
        b = (rng.integers(-64, 64, size=(K, N)) / 64.0 * 2.0 ** -30).astype(np.float32)
        for _ in range(int(rng.integers(1, 3))):
            a[rng.integers(M), rng.integers(K)] = big[rng.integers(len(big))]
        c = (rng.integers(-64, 64, size=(M, N)) / 64.0).astype(np.float32)
        alpha, beta = [(1.0, 0.0), (1.5, -0.5), (-0.75, 2.0)][trial % 3]
        out = oracle.sgemm("N", "N", a, b, c, alpha, beta, lib=lib)
        for i in range(M):
            for j in range(N):
                exact = Fraction(alpha) * sum(Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(K))
                if beta != 0.0:
                    exact += Fraction(beta) * Fraction(float(c[i, j]))
                assert out[i, j] == _round_f32(exact), (trial, i, j, out[i, j], float(exact))


def pin_ieee_special_values(lib):
    """IEEE 754: Inf * finite = +-Inf with the product's sign, Inf * 0 = NaN, Inf - Inf = NaN,
    NaN propagates; beta * C with Inf in C gives Inf, beta = 0 leaves C unread."""
    inf, nan = np.inf, np.nan
    cases = [  # (a row, b column, expected a.b)
        ([inf, 1.0], [2.0, 3.0], inf),
        ([inf, 1.0], [-2.0, 3.0], -inf),
        ([-inf, 1.0], [-0.5, 3.0], inf),
        ([inf, 1.0], [0.0, 3.0], nan),
        ([0.0, 1.0], [inf, 3.0], nan),
        ([inf, -inf], [1.0, 1.0], nan),
        ([inf, inf], [1.0, 2.0], inf),
        ([nan, 1.0], [0.0, 3.0], nan),
        ([1.0, 2.0], [3.0, -inf], -inf),
        ([2.0 ** 100, 2.0 ** 100], [2.0 ** 27, 2.0 ** 27], inf),  # the float32 result overflows
    ]
    for arow, bcol, want in cases:
        a = np.array([arow], np.float32)
        b = np.array(bcol, np.float32).reshape(2, 1)
        got = oracle.sgemm("N", "N", a, b, lib=lib)[0, 0]
        assert (np.isnan(want) and np.isnan(got)) or got == want, (arow, bcol, got)
    a = np.ones((1, 1), np.float32)
    c = np.array([[inf]], np.float32)
    assert oracle.sgemm("N", "N", a, a, c, 1.0, -0.5, lib=lib)[0, 0] == -inf
    assert oracle.sgemm("N", "N", a, a, c, 1.0, 0.0, lib=lib)[0, 0] == 1.0


def _nearer(x, t, u, tie_to_t):
    """Of the candidates t (toward zero) and u (away from zero) around finite x, the nearer one;
    a tie goes to u unless tie_to_t.  A u of +-Inf stands for the value 2^128 just past the top of
    the format (rounding there overflows to +-Inf), so distances use that value."""
    x64, t64 = x.astype(np.float64), t.astype(np.float64)
    u64 = np.where(np.isinf(u), np.copysign(2.0 ** 128, x64), u.astype(np.float64))
    dt, du = np.abs(x64 - t64), np.abs(u64 - x64)
    return np.where((dt < du) | ((dt == du) & tie_to_t), t, u).astype(np.float32)


def _tf32_by_bits(x: np.ndarray) -> np.ndarray:
    """TF32 rounding characterized on the bits, independently of the oracle's arithmetic: the
    candidates are x with its 13 low fraction bits cleared (t, toward zero) and the next TF32
    value above it in magnitude (t + 2^13 ulps); the result is the nearer one, the larger
    magnitude on a tie (ties away from zero).  Finite x only."""
    x = np.asarray(x, np.float32)
    b = x.view(np.uint32)
    t = (b & np.uint32(0xFFFFE000)).view(np.float32)
    u = ((b & np.uint32(0xFFFFE000)) + np.uint32(0x2000)).view(np.float32)  # +-Inf at the top
    return _nearer(x, t, u, np.zeros(x.shape, bool))


def pin_tf32_round_golden(lib):
    """The hand-worked TF32 roundings of tests/golden/tf32_round.txt, and NaN stays NaN."""
    rows = []
    with open(os.path.join(GOLDEN, "tf32_round.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                x, y = line.split()[:2]
                rows.append((int(x, 16), int(y, 16)))
    x = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    want = np.array([r[1] for r in rows], np.uint32)
    got = oracle.round_tf32(x, lib).view(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(rows[i][0]), hex(int(got[i])), hex(rows[i][1])) for i in bad]
    assert np.isnan(oracle.round_tf32(np.array([np.nan, -np.nan], np.float32), lib)).all()


def pin_tf32_round_properties(lib):
    """Finite floats over the whole exponent range (normal and subnormal, both signs): the result
    is a TF32 value (13 low fraction bits zero, or +-Inf past the top) and equals the bit-level
    characterization above."""
    rng = np.random.default_rng(18)
    bits = rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.round_tf32(x, lib)
    fin = np.isfinite(got)
    assert np.all((got[fin].view(np.uint32) & np.uint32(0x1FFF)) == 0)
    assert np.array_equal(got.view(np.uint32), _tf32_by_bits(x).view(np.uint32))


def pin_tf32_gemm(lib):
    """The TF32-input GEMM: inputs that are already TF32 values give the FP32 oracle's result;
    on tiny shapes with 12-bit dyadic inputs (which the rounding changes) it equals a float64
    einsum of the bit-level-rounded inputs, rounded once (every product and sum exact)."""
    rng = np.random.default_rng(19)
    for (ta, tb), M, N, K in itertools.product(OPS, (1, 3, 7), (2, 5), (1, 4, 9)):
        A = _stored(rng, ta, M, K, dyadic_bits=6)
        B = _stored(rng, tb, K, N, dyadic_bits=6)
        C = _stored(rng, "N", M, N, dyadic_bits=6)
        assert np.array_equal(oracle.sgemm_tf32(ta, tb, A, B, C, 1.5, -0.5, lib=lib),
                              oracle.sgemm(ta, tb, A, B, C, 1.5, -0.5, lib=lib)), (ta, tb, M, N, K)
        A = _stored(rng, ta, M, K, dyadic_bits=12)
        B = _stored(rng, tb, K, N, dyadic_bits=12)
        ref = (1.5 * np.einsum("ik,kj->ij", _op(_tf32_by_bits(A), ta).astype(np.float64),
                               _op(_tf32_by_bits(B), tb).astype(np.float64))
               - 0.5 * C.astype(np.float64)).astype(np.float32)
        got = oracle.sgemm_tf32(ta, tb, A, B, C, 1.5, -0.5, lib=lib)
        assert np.array_equal(got, ref), (ta, tb, M, N, K)
    # the rounding really happens: 1 + 2^-11 (a tie) times 1 gives 1 + 2^-10
    a = np.array([[1 + 2.0 ** -11]], np.float32)
    assert oracle.sgemm_tf32("N", "N", a, np.ones((1, 1), np.float32), lib=lib)[0, 0] == np.float32(1 + 2.0 ** -10)


def _bf16_by_bits(x: np.ndarray) -> np.ndarray:
    """BF16 rounding characterized on the bits, independently of the oracle's arithmetic: the
    candidates are x with its 16 low bits cleared (t, toward zero) and the next BF16 value above
    it in magnitude (t + 2^16 ulps); the result is the nearer one, on a tie the one whose lowest
    kept bit (bit 16) is 0.  Finite x only."""
    x = np.asarray(x, np.float32)
    b = x.view(np.uint32)
    tb = b & np.uint32(0xFFFF0000)
    ub = tb + np.uint32(0x10000)  # +-Inf at the top
    return _nearer(x, tb.view(np.float32), ub.view(np.float32), (tb & np.uint32(0x10000)) == 0)


def pin_bf16_round_golden(lib):
    """The hand-worked BF16 roundings of tests/golden/bf16_round.txt, and NaN stays NaN."""
    rows = []
    with open(os.path.join(GOLDEN, "bf16_round.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                x, y = line.split()[:2]
                rows.append((int(x, 16), int(y, 16)))
    x = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    want = np.array([r[1] for r in rows], np.uint32)
    got = oracle.round_bf16(x, lib).view(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(rows[i][0]), hex(int(got[i])), hex(rows[i][1])) for i in bad]
    assert np.isnan(oracle.round_bf16(np.array([np.nan, -np.nan], np.float32), lib)).all()


def pin_bf16_round_properties(lib):
    """Finite floats over the whole exponent range (normal and subnormal, both signs): the result
    is a BF16 value (16 low bits zero, or +-Inf past the top) and equals the bit-level
    characterization above."""
    rng = np.random.default_rng(20)
    bits = rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    # and exact ties: a kept pattern followed by exactly half a quantum
    ties = (rng.integers(0, 1 << 16, size=20000, dtype=np.uint64).astype(np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    x = np.concatenate([bits, ties]).view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.round_bf16(x, lib)
    fin = np.isfinite(got)
    assert np.all((got[fin].view(np.uint32) & np.uint32(0xFFFF)) == 0)
    assert np.array_equal(got.view(np.uint32), _bf16_by_bits(x).view(np.uint32))


def pin_bf16_gemm(lib):
    """The BF16-input GEMM: inputs that are already BF16 values give the FP32 oracle's result; on
    tiny shapes with 12-bit dyadic inputs (which the rounding changes) it equals a float64 einsum
    of the bit-level-rounded inputs, rounded once (every product and sum exact)."""
    rng = np.random.default_rng(21)
    for (ta, tb), M, N, K in itertools.product(OPS, (1, 3, 7), (2, 5), (1, 4, 9)):
        A = _stored(rng, ta, M, K, dyadic_bits=6)
        B = _stored(rng, tb, K, N, dyadic_bits=6)
        C = _stored(rng, "N", M, N, dyadic_bits=6)
        assert np.array_equal(oracle.sgemm_bf16(ta, tb, A, B, C, 1.5, -0.5, lib=lib),
                              oracle.sgemm(ta, tb, A, B, C, 1.5, -0.5, lib=lib)), (ta, tb, M, N, K)
        A = _stored(rng, ta, M, K, dyadic_bits=12)
        B = _stored(rng, tb, K, N, dyadic_bits=12)
        ref = (1.5 * np.einsum("ik,kj->ij", _op(_bf16_by_bits(A), ta).astype(np.float64),
                               _op(_bf16_by_bits(B), tb).astype(np.float64))
               - 0.5 * C.astype(np.float64)).astype(np.float32)
        got = oracle.sgemm_bf16(ta, tb, A, B, C, 1.5, -0.5, lib=lib)
        assert np.array_equal(got, ref), (ta, tb, M, N, K)
    # the rounding really happens: 1 + 3 * 2^-8 (a tie, to even) times 1 gives 1 + 2^-6
    a = np.array([[1 + 3 * 2.0 ** -8]], np.float32)
    assert oracle.sgemm_bf16("N", "N", a, np.ones((1, 1), np.float32), lib=lib)[0, 0] == np.float32(1 + 2.0 ** -6)


ALL_PINS = [
    pin_hand_2x2, pin_bruteforce_tiny, pin_integer_pattern, pin_integer_alpha_beta, pin_k1_exact,
    pin_alpha_zero, pin_k_zero, pin_beta_zero_nan_c, pin_identity, pin_transpose_identity,
    pin_transposed_copy, pin_alpha_pow2, pin_padding_not_read, pin_random_vs_float64_matmul,
    pin_bound_magnitude, pin_argument_errors, pin_conjugate_is_transpose, pin_batched_dyadic,
    pin_batched_edges, pin_large_finite_exact, pin_ieee_special_values, pin_tf32_round_golden,
    pin_tf32_round_properties, pin_tf32_gemm, pin_bf16_round_golden, pin_bf16_round_properties, pin_bf16_gemm,
]
