"""Python binding of libsgemm (C ABI in include/sgemm.h): argument marshalling only.

Every entry point of the C library is exposed under the same name.  Matrix
arguments may be raw device addresses (int), torch CUDA tensors (their
``data_ptr()`` is passed) or None (NULL).  ``stream`` may be None (torch's
current stream), an int handle, or a ``torch.cuda.Stream``.  All arithmetic
runs in the library's CUDA kernels; there is no fallback: if the compiled
library is missing, ``load()`` raises.

    C = alpha * op(A) * op(B) + beta * C     (row-major float32, op = N or T)
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SgemmError", "load", "library_path", "sgemm", "sgemm_host", "sgemm_noalloc", "sgemm_ex",
    "sgemm_workspace_size", "sgemm_plan",
    "sgemm_strided_batched", "sgemm_plan_strided_batched", "sgemm_status_string",
    "sgemm_last_cuda_error", "sgemm_sync_status", "sgemm_set_variant_override",
    "sgemm_selftest_wait_timeout", "matmul", "VARIANTS", "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libsgemm.so")

STATUS = {"OK": 0, "ERR_CUDA": 1, "ERR_TIMEOUT": 2, "ERR_NOMEM": 3, "ERR_UNSUPPORTED": 4, "ERR_SCRATCH_LIMIT": 5,
          "ERR_BOUNDS": 6}
NOALLOC_SCRATCH_BYTES = 32 << 20  # SGEMM_NOALLOC_SCRATCH_BYTES in include/sgemm.h
VARIANTS = {"AUTO": 0, "NONE": 1, "SCALE": 2, "GENERIC": 3, "TMA_128x128": 4, "TMA_64x256": 5, "TC_TF32X3": 6,
            "SMALL": 7, "TC_GROUPED": 8, "TC_PAIR": 9,
            "TC_PRESPLIT": 10, "TC_TF32": 11, "TC_SKINNY": 12,
            "TC_BF16": 13}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str = "sgemm"):
        self.status = status
        # the failed CUDA call's cudaError_t (kept per host thread; raised on the caller's thread)
        self.cuda_error = sgemm_last_cuda_error() if status == STATUS["ERR_CUDA"] else 0
        detail = f" (cudaError_t {self.cuda_error})" if self.cuda_error else ""
        super().__init__(f"{where} returned {status}: {sgemm_status_string(status)}{detail}")


class PlanStruct(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("stages", ctypes.c_int), ("threads", ctypes.c_int),
                ("split_k", ctypes.c_int), ("kernel_launches", ctypes.c_int),
                ("grid_x", ctypes.c_int64), ("grid_y", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
                ("dp_tiles", ctypes.c_int64), ("sk_tiles", ctypes.c_int64), ("sk_iters", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """C signatures of the exported entry points."""
    i64, f32, vp, ch = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_char
    lib.sgemm.restype = ctypes.c_int
    lib.sgemm.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm_host.restype = ctypes.c_int
    lib.sgemm_host.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm_noalloc.restype = ctypes.c_int
    lib.sgemm_noalloc.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm_ex.restype = ctypes.c_int
    lib.sgemm_ex.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp, ctypes.c_size_t, vp]
    lib.sgemm_workspace_size.restype = ctypes.c_int
    lib.sgemm_workspace_size.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.sgemm_plan.restype = ctypes.c_int
    lib.sgemm_plan.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, ctypes.c_int,
                               ctypes.POINTER(PlanStruct)]
    lib.sgemm_plan_for_device.restype = ctypes.c_int
    lib.sgemm_plan_for_device.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                          ctypes.c_int, ctypes.c_int, ctypes.POINTER(PlanStruct)]
    lib.sgemm_release_workspace.restype = ctypes.c_int
    lib.sgemm_release_workspace.argtypes = [ctypes.c_size_t]
    lib.sgemm_clock_snapshot.restype = ctypes.c_int
    lib.sgemm_clock_snapshot.argtypes = [vp, ctypes.c_int, vp]
    lib.sgemm_bf16.restype = ctypes.c_int
    lib.sgemm_bf16.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm_bf16_plan.restype = ctypes.c_int
    lib.sgemm_bf16_plan.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, ctypes.c_int,
                                    ctypes.POINTER(PlanStruct)]
    lib.sgemm_tf32.restype = ctypes.c_int
    lib.sgemm_tf32.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.sgemm_tf32_plan.restype = ctypes.c_int
    lib.sgemm_tf32_plan.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, ctypes.c_int,
                                    ctypes.POINTER(PlanStruct)]
    lib.sgemm_strided_batched.restype = ctypes.c_int
    lib.sgemm_strided_batched.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                          i64, i64, i64, i64, vp]
    lib.sgemm_plan_strided_batched.restype = ctypes.c_int
    lib.sgemm_plan_strided_batched.argtypes = [ch, ch, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                               i64, i64, i64, i64, ctypes.c_int, ctypes.POINTER(PlanStruct)]
    lib.sgemm_status_string.restype = ctypes.c_char_p
    lib.sgemm_status_string.argtypes = [ctypes.c_int]
    lib.sgemm_last_cuda_error.restype = ctypes.c_int
    lib.sgemm_last_cuda_error.argtypes = []
    lib.sgemm_sync_status.restype = ctypes.c_int
    lib.sgemm_sync_status.argtypes = [vp]
    lib.sgemm_set_variant_override.restype = ctypes.c_int
    lib.sgemm_set_variant_override.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.sgemm_selftest_wait_timeout.restype = ctypes.c_int
    lib.sgemm_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.sgemm_bounds_report.restype = ctypes.c_int
    lib.sgemm_bounds_report.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_longlong)]
    lib.sgemm_debug_bounds_enabled.restype = ctypes.c_int
    lib.sgemm_debug_bounds_enabled.argtypes = []
    lib.sgemm_selftest_bounds.restype = ctypes.c_int
    lib.sgemm_selftest_bounds.argtypes = [vp]
    return lib


def load() -> ctypes.CDLL:
    """Load the compiled libsgemm.so (build it with ``python -m sgemm_row_major_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libsgemm.so not built: {_LIB_PATH} is missing "
                              "(run `python -m sgemm_row_major_gb300.build`)")
        _lib = _declare(ctypes.CDLL(_LIB_PATH))
        return _lib


def load_debug() -> ctypes.CDLL:
    """The bounds-checking build libsgemm_debug.so (``python -m sgemm_row_major_gb300.build --debug``),
    loaded beside libsgemm.so with the same entry points; its kernels check every index."""
    path = os.path.join(os.path.dirname(_LIB_PATH), "libsgemm_debug.so")
    if not os.path.exists(path):
        raise ImportError(f"libsgemm_debug.so not built: {path} is missing "
                          "(run `python -m sgemm_row_major_gb300.build --debug`)")
    return _declare(ctypes.CDLL(path))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not getattr(x, "is_cuda", False):
            raise TypeError("sgemm operands must be CUDA tensors or device addresses")
        return int(x.data_ptr())
    raise TypeError(f"cannot pass {type(x).__name__} as a device pointer")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) or None
    if isinstance(s, int):
        return s or None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream) or None
    raise TypeError("stream must be None, an int handle or a torch.cuda.Stream")


def _ch(t) -> bytes:
    if isinstance(t, bytes):
        return t[:1]
    return str(t).encode()[:1]


def sgemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, *,
          raise_on_error: bool = True) -> int:
    """C = alpha*op(A)*op(B) + beta*C, row-major float32 on the device (see include/sgemm.h).

    Returns the C status (0 on success); raises SgemmError on a nonzero status
    unless ``raise_on_error=False``.
    """
    st = load().sgemm(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                      _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st)
    return st


def _host_ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if getattr(x, "is_cuda", False):
            raise TypeError("sgemm_host operands must be host memory")
        return int(x.data_ptr())
    if hasattr(x, "__array_interface__"):
        return int(x.__array_interface__["data"][0])
    raise TypeError(f"cannot pass {type(x).__name__} as a host pointer")


def sgemm_host(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, *,
               raise_on_error: bool = True) -> int:
    """sgemm() on HOST operands (numpy arrays, CPU tensors or addresses); C is written back to host memory.

    Asynchronous on ``stream``: synchronise it before reading C.  Page-locked
    host memory (e.g. ``torch.empty(..., pin_memory=True)``) gives full speed.
    """
    st = load().sgemm_host(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _host_ptr(A),
                           int(lda), _host_ptr(B), int(ldb), float(beta), _host_ptr(C), int(ldc), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_host")
    return st


def sgemm_noalloc(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, *,
                  raise_on_error: bool = True) -> int:
    """sgemm() for callers that cannot allocate device memory during the call.

    Same arguments and results as sgemm(); split-K partial sums go to a fixed
    32 MiB array inside the library instead of a memory pool.  Problems that
    need more scratch return ERR_SCRATCH_LIMIT.  All calls on a device share
    that array, so calls that can overlap on the GPU must be ordered.
    """
    st = load().sgemm_noalloc(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                              int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_noalloc")
    return st


def sgemm_workspace_size(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) -> int:
    """Bytes of workspace sgemm_ex() needs for these arguments on the current device (0: none)."""
    n = ctypes.c_size_t(0)
    st = load().sgemm_workspace_size(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                     int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), ctypes.byref(n))
    if st != 0:
        raise SgemmError(st, "sgemm_workspace_size")
    return int(n.value)


def sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace, workspace_bytes,
             stream=None, *, raise_on_error: bool = True) -> int:
    """sgemm() with the split-K partial sums in a caller-owned device workspace (16-byte aligned, at
    least sgemm_workspace_size() bytes; None when that is 0): no allocation, no size limit."""
    st = load().sgemm_ex(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                         _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _ptr(workspace), int(workspace_bytes),
                         _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_ex")
    return st


def sgemm_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, sm_count: int = 0) -> dict:
    """The launch sgemm() would make (pure host logic when sm_count > 0).  Raises on invalid arguments."""
    plan = PlanStruct()
    st = load().sgemm_plan(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                           _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), int(sm_count), ctypes.byref(plan))
    if st != 0:
        raise SgemmError(st, "sgemm_plan")
    out = {name: getattr(plan, name) for name, _ in PlanStruct._fields_}
    out["variant_name"] = VARIANT_NAMES.get(out["variant"], str(out["variant"]))
    return out


def sgemm_plan_for_device(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, sm_count: int,
                          pair_clusters: int) -> dict:
    """The launch sgemm() would make on a device of sm_count SMs holding pair_clusters CTA-pair
    clusters at once (0: none).  Pure host logic.  Raises on invalid arguments."""
    plan = PlanStruct()
    st = load().sgemm_plan_for_device(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                      int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), int(sm_count),
                                      int(pair_clusters), ctypes.byref(plan))
    if st != 0:
        raise SgemmError(st, "sgemm_plan_for_device")
    out = {name: getattr(plan, name) for name, _ in PlanStruct._fields_}
    out["variant_name"] = VARIANT_NAMES.get(out["variant"], str(out["variant"]))
    return out


def sgemm_release_workspace(keep_bytes: int = 0) -> None:
    """Return pooled workspace memory of the current device beyond keep_bytes to the driver."""
    st = load().sgemm_release_workspace(int(keep_bytes))
    if st != 0:
        raise SgemmError(st, "sgemm_release_workspace")


def sgemm_tf32(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, *,
               raise_on_error: bool = True) -> int:
    """C = alpha*op(tf32(A))*op(tf32(B)) + beta*C: inputs rounded to TF32 (nearest, ties away),
    FP32 accumulation on the tensor cores."""
    st = load().sgemm_tf32(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                           _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_tf32")
    return st


def sgemm_tf32_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, sm_count: int = 0) -> dict:
    """The launch sgemm_tf32() would make.  Raises on invalid arguments."""
    plan = PlanStruct()
    st = load().sgemm_tf32_plan(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                                _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), int(sm_count), ctypes.byref(plan))
    if st != 0:
        raise SgemmError(st, "sgemm_tf32_plan")
    out = {name: getattr(plan, name) for name, _ in PlanStruct._fields_}
    out["variant_name"] = VARIANT_NAMES.get(out["variant"], str(out["variant"]))
    return out


def sgemm_bf16(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, *,
               raise_on_error: bool = True) -> int:
    """C = alpha*op(bf16(A))*op(bf16(B)) + beta*C: inputs rounded to BF16 (nearest, ties to even),
    FP32 accumulation on the tensor cores."""
    st = load().sgemm_bf16(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                           _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_bf16")
    return st


def sgemm_bf16_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, sm_count: int = 0) -> dict:
    """The launch sgemm_bf16() would make.  Raises on invalid arguments."""
    plan = PlanStruct()
    st = load().sgemm_bf16_plan(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                                _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), int(sm_count), ctypes.byref(plan))
    if st != 0:
        raise SgemmError(st, "sgemm_bf16_plan")
    out = {name: getattr(plan, name) for name, _ in PlanStruct._fields_}
    out["variant_name"] = VARIANT_NAMES.get(out["variant"], str(out["variant"]))
    return out


def sgemm_clock_snapshot(out, stream=None) -> None:
    """Per-SM (cycle counter, global ns timer) pairs into `out`, a CUDA int64 tensor of 2 * slots
    elements (slot = SM id), enqueued on `stream`."""
    st = load().sgemm_clock_snapshot(_ptr(out), int(out.numel()) // 2, _stream(stream))
    if st != 0:
        raise SgemmError(st, "sgemm_clock_snapshot")


def sgemm_strided_batched(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                          strideA, strideB, strideC, batch_count, stream=None, *, raise_on_error: bool = True) -> int:
    """batch_count products C_b = alpha*op(A_b)*op(B_b) + beta*C_b with X_b = X + b*strideX (elements)."""
    st = load().sgemm_strided_batched(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                      int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), int(strideA),
                                      int(strideB), int(strideC), int(batch_count), _stream(stream))
    if st != 0 and raise_on_error:
        raise SgemmError(st, "sgemm_strided_batched")
    return st


def sgemm_plan_strided_batched(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                               strideA, strideB, strideC, batch_count, sm_count: int = 0) -> dict:
    """The launch sgemm_strided_batched() would make.  Raises on invalid arguments."""
    plan = PlanStruct()
    st = load().sgemm_plan_strided_batched(_ch(transA), _ch(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                           int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc),
                                           int(strideA), int(strideB), int(strideC), int(batch_count),
                                           int(sm_count), ctypes.byref(plan))
    if st != 0:
        raise SgemmError(st, "sgemm_plan_strided_batched")
    out = {name: getattr(plan, name) for name, _ in PlanStruct._fields_}
    out["variant_name"] = VARIANT_NAMES.get(out["variant"], str(out["variant"]))
    return out


def sgemm_status_string(status: int) -> str:
    return load().sgemm_status_string(int(status)).decode()


def sgemm_last_cuda_error() -> int:
    return int(load().sgemm_last_cuda_error())


def sgemm_sync_status(stream=None) -> int:
    return int(load().sgemm_sync_status(_stream(stream)))


def sgemm_set_variant_override(variant, split_k: int = 0) -> None:
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    st = load().sgemm_set_variant_override(v, int(split_k))
    if st != 0:
        raise SgemmError(st, "sgemm_set_variant_override")


def sgemm_selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    return int(load().sgemm_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def _stored_ld(X, name: str) -> int:
    import torch
    if X.dim() != 2 or X.dtype != torch.float32:
        raise TypeError(f"{name} must be a 2-D float32 tensor")
    if X.shape[1] > 1 and X.stride(1) != 1:
        raise TypeError(f"{name} rows must be contiguous (stride(1) == 1)")
    return max(int(X.stride(0)) if X.shape[0] > 1 else int(X.shape[1]), 1)


def matmul(A, B, C=None, transA: str = "N", transB: str = "N", alpha: float = 1.0, beta: float = 0.0,
           stream=None):
    """Tensor convenience: derives M, N, K and the leading dimensions from 2-D CUDA tensors.

    A and B are the STORED matrices (A is M x K for 'N', K x M for 'T'; likewise
    B).  C (M x N) is updated in place and returned; when C is None a new
    tensor is allocated and beta must be 0.
    """
    import torch
    ta, tb = transA.upper() in ("T", "C"), transB.upper() in ("T", "C")
    M = A.shape[1] if ta else A.shape[0]
    K = A.shape[0] if ta else A.shape[1]
    N = B.shape[0] if tb else B.shape[1]
    if (B.shape[1] if tb else B.shape[0]) != K:
        raise ValueError("inner dimensions of op(A) and op(B) differ")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if tuple(C.shape) != (M, N):
        raise ValueError("C has the wrong shape")
    sgemm(transA, transB, M, N, K, alpha, A, _stored_ld(A, "A"), B, _stored_ld(B, "B"), beta, C,
          _stored_ld(C, "C"), stream)
    return C
