"""CPU oracle for row-major SGEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library (``sgemm_row_major_gb300``) never imports it, and it never imports the
CUDA library.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, double accumulation); this
module only compiles it with gcc and marshals numpy arrays through ctypes.

Definition followed (itan.pw "CUDA NVIDIA 4090 高性能計算", 概要, and
klklkl10086.github.io "Sgemm单精度矩阵乘法", 问题定义)::

    Cref_ij = fl32(alpha * sum_k op(A)_ik op(B)_kj + beta * C_ij)   (in double)

Also the TF32-input GEMM: A and B rounded to TF32 (round_tf32, ties away
from zero), then the same SGEMM; and the BF16-input GEMM: A and B rounded to
BF16 (round_bf16, ties to even), then the same SGEMM.

Pins (tests/test_oracle.py): the 2MNK FLOP count the pages print, brute force
against an independent float64 einsum on tiny shapes, exact integer results on
the pages' (j-i)%3 pattern against an int64 matmul, the K=1 correctly rounded
product, alpha=0 -> beta*C, identity -> alpha*B + beta*C, (AB)^T = B^T A^T,
op='T' on a transposed copy, exact power-of-two scaling of alpha, and the
bound magnitude S against |A|@|B|; the strided batch against a float64 einsum
over stacked dyadic operands, with shared (stride 0) operands and NaN gaps
between matrices.  tests/test_oracle_mutations.py plants
mistakes in a copy of the C source and checks that a pin catches each one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(_BUILD_DIR, "liboracle_sgemm.so")

# -ffp-contract=off and no -ffast-math: the compiler may not fuse or reorder
# the double arithmetic of the oracle.
CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", "-std=c11"]

_lock = threading.Lock()
_lib = None


def compile_library(source: str = SOURCE, output: str = LIBRARY, extra_flags=()) -> str:
    """Compile an oracle C source into a shared library with gcc; returns its path."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra_flags, source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, output)
    return output


def build(force: bool = False) -> str:
    """Build liboracle_sgemm.so if it is missing or older than its source."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_library()
    return LIBRARY


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_sgemm
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_char, ctypes.c_char, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64]
    g = lib.oracle_sgemm_strided_batched
    g.restype = ctypes.c_int
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    g.argtypes = [ctypes.c_char, ctypes.c_char, i64, i64, i64,
                  ctypes.c_float, vp, i64, i64,
                  vp, i64, i64,
                  ctypes.c_float, vp, i64, i64,
                  i64, vp, i64, i64]
    lib.oracle_round_tf32.restype = None
    lib.oracle_round_tf32.argtypes = [vp, vp, i64]
    lib.oracle_round_bf16.restype = None
    lib.oracle_round_bf16.argtypes = [vp, vp, i64]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _library() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def set_num_threads(n: int) -> None:
    """Threads later oracle calls use (the arithmetic of an element does not depend on it)."""
    _library().oracle_set_num_threads(int(n))


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loop uses (OMP_NUM_THREADS or all cores)."""
    return int(_library().oracle_num_threads())


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


class OracleError(ValueError):
    pass


def sgemm_raw(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, S=None, lds=0, lib=None) -> int:
    """Call the C oracle on flat float32 buffers; C (and S) are updated in place.

    A, B, C are 1-D float32 numpy arrays holding the stored matrices with row
    strides lda, ldb, ldc (elements).  Returns the oracle's status (0 or -i).
    """
    lib = lib or _library()
    for name, arr, dt in (("A", A, np.float32), ("B", B, np.float32), ("C", C, np.float32)):
        if arr is not None and (arr.dtype != dt or not arr.flags.c_contiguous):
            raise OracleError(f"{name} must be a C-contiguous float32 array")
    if S is not None and (S.dtype != np.float64 or not S.flags.c_contiguous):
        raise OracleError("S must be a C-contiguous float64 array")
    return int(lib.oracle_sgemm(_c(transA), _c(transB), int(M), int(N), int(K),
                                float(alpha), _ptr(A), int(lda), _ptr(B), int(ldb),
                                float(beta), _ptr(C), int(ldc), _ptr(S), int(lds)))


def sgemm_strided_batched(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                          strideC, batch, want_bound: bool = False, lib=None):
    """Strided batch on flat float32 buffers: product b reads A[b*strideA:],
    B[b*strideB:] and updates C[b*strideC:] (see oracle_sgemm_strided_batched).

    Returns a new flat C buffer (the input C is not modified) and, with
    ``want_bound``, S as a (batch, M, N) float64 array.
    """
    lib = lib or _library()
    for name, arr in (("A", A), ("B", B), ("C", C)):
        if arr is not None and (arr.dtype != np.float32 or arr.ndim != 1 or not arr.flags.c_contiguous):
            raise OracleError(f"{name} must be a flat C-contiguous float32 array")
    out = None if C is None else C.copy()
    S = np.zeros((max(int(batch), 0), int(M), int(N)), dtype=np.float64) if want_bound else None
    st = int(lib.oracle_sgemm_strided_batched(
        _c(transA), _c(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), int(strideA),
        _ptr(B), int(ldb), int(strideB), float(beta), _ptr(out), int(ldc), int(strideC), int(batch),
        _ptr(S), int(N), int(M) * int(N)))
    if st != 0:
        raise OracleError(f"oracle_sgemm_strided_batched returned {st}")
    return (out, S) if want_bound else out


def _c(t) -> bytes:
    return t.encode() if isinstance(t, str) else bytes(t)


def sgemm(transA: str, transB: str, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
          alpha: float = 1.0, beta: float = 0.0, M: int | None = None, N: int | None = None,
          K: int | None = None, want_bound: bool = False, lib=None):
    """Oracle SGEMM on 2-D row-major float32 arrays holding the STORED matrices.

    A is M x K for 'N' or K x M for 'T' (likewise B is K x N or N x K); the
    row stride of each array (its leading dimension) may exceed its logical
    width: pass a slice ``X[:, :cols]`` of a wider array, or M/N/K explicitly.
    C (M x N, may be None when beta == 0) is not modified.  Returns the new C
    as a float32 array, and S (float64, M x N) when ``want_bound``.
    """
    ta = transA.upper() in ("T", "C")
    tb = transB.upper() in ("T", "C")
    if M is None:
        M = A.shape[1] if ta else A.shape[0]
    if K is None:
        K = A.shape[0] if ta else A.shape[1]
    if N is None:
        N = B.shape[0] if tb else B.shape[1]
    a_flat, lda = _flat_view(A)
    b_flat, ldb = _flat_view(B)
    out = np.zeros((M, N), dtype=np.float32) if C is None else np.array(C[:M, :N], dtype=np.float32, copy=True)
    if C is None and beta != 0.0:
        raise OracleError("beta != 0 needs C")
    S = np.zeros((M, N), dtype=np.float64) if want_bound else None
    st = sgemm_raw(transA, transB, M, N, K, alpha, a_flat, lda, b_flat, ldb, beta,
                   out.reshape(-1) if out.size else np.zeros(1, np.float32), max(N, 1),
                   None if S is None else (S.reshape(-1) if S.size else np.zeros(1, np.float64)),
                   max(N, 1), lib=lib)
    if st != 0:
        raise OracleError(f"oracle rejected argument {-st}")
    return (out, S) if want_bound else out


def _flat_view(X: np.ndarray):
    """(flat float32 buffer, row stride) for a 2-D array whose rows may be strided."""
    if X.dtype != np.float32:
        raise OracleError("operands must be float32")
    if X.ndim != 2:
        raise OracleError("operands must be 2-D")
    rows, cols = X.shape
    if X.size == 0:
        return np.zeros(1, np.float32), max(cols, 1)
    if X.strides[1] != 4 and cols > 1:
        raise OracleError("operand rows must be contiguous")
    ld = X.strides[0] // 4 if rows > 1 else max(cols, 1)
    if X.flags.c_contiguous:
        return X.reshape(-1) if X.size else np.zeros(1, np.float32), max(ld, 1)
    # a column-slice of a wider row-major array: view the whole underlying span
    span = (rows - 1) * ld + cols
    flat = np.lib.stride_tricks.as_strided(X, shape=(span,), strides=(4,))
    return np.ascontiguousarray(flat), ld


def round_tf32(x: np.ndarray, lib=None) -> np.ndarray:
    """x (float32) rounded to TF32 -- 10 fraction bits, to nearest with ties away from zero;
    past FLT_MAX to +-Inf; +-0, +-Inf, NaN kept -- by the C oracle's rounding (a new array)."""
    lib = lib or _library()
    src = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(src)
    if src.size:
        lib.oracle_round_tf32(src.ctypes.data, out.ctypes.data, src.size)
    return out


def round_bf16(x: np.ndarray, lib=None) -> np.ndarray:
    """x (float32) rounded to BF16 -- 7 fraction bits, to nearest with ties to even; past the
    largest BF16 value to +-Inf; +-0, +-Inf, NaN kept -- by the C oracle's rounding, returned as
    float32 (a new array)."""
    lib = lib or _library()
    src = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(src)
    if src.size:
        lib.oracle_round_bf16(src.ctypes.data, out.ctypes.data, src.size)
    return out


def sgemm_bf16(transA: str, transB: str, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
               alpha: float = 1.0, beta: float = 0.0, M: int | None = None, N: int | None = None,
               K: int | None = None, want_bound: bool = False, lib=None):
    """The BF16-input GEMM: oracle SGEMM (sgemm above) on the stored A and B rounded to BF16
    (round_bf16); C, alpha, beta as they are.  S, when wanted, is that of the rounded inputs."""
    return sgemm(transA, transB, round_bf16(A, lib), round_bf16(B, lib), C, alpha, beta, M=M, N=N, K=K,
                 want_bound=want_bound, lib=lib)


def sgemm_tf32(transA: str, transB: str, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
               alpha: float = 1.0, beta: float = 0.0, M: int | None = None, N: int | None = None,
               K: int | None = None, want_bound: bool = False, lib=None):
    """The TF32-input GEMM: oracle SGEMM (sgemm above) on the stored A and B rounded to TF32
    (round_tf32); C, alpha, beta as they are.  S, when wanted, is that of the rounded inputs."""
    return sgemm(transA, transB, round_tf32(A, lib), round_tf32(B, lib), C, alpha, beta, M=M, N=N, K=K,
                 want_bound=want_bound, lib=lib)
