"""Build libsgemm.so in-tree with nvcc for sm_103a.

Each .cu translation unit under csrc/ compiles in parallel to an object file
under _build/, and nvcc links them into ``_lib/libsgemm.so`` (CUDA runtime
linked statically, no dependency on torch).  Usage: ``python -m
sgemm_row_major_gb300.build`` or ``build()`` from Python.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIBRARY = os.path.join(LIB_DIR, "libsgemm.so")
# the same sources with the kernels' bounds checks compiled in (-DSGEMM_DEBUG_BOUNDS)
DEBUG_LIBRARY = os.path.join(LIB_DIR, "libsgemm_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsgemm")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def source_digest() -> str:
    """Hash of every source and header of the library (identifies a kernel build)."""
    h = hashlib.sha256()
    for path in sources() + _headers():
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TMA_KERNEL_FILES = ["kernel_tma.cuh", "device_utils.cuh", "sgemm_internal.h", "kernel_tma_nn.cu",
                    "kernel_tma_nt.cu", "kernel_tma_tn.cu", "kernel_tma_tt.cu"]


TC_KERNEL_FILES = ["kernel_tf32x3.cu", "kernel_tc_common.cuh", "device_utils.cuh", "sgemm_internal.h"]


PAIR_KERNEL_FILES = ["kernel_tc_pair.cu", "kernel_tc_common.cuh", "device_utils.cuh", "sgemm_internal.h"]


PRESPLIT_KERNEL_FILES = ["kernel_presplit.cu", "kernel_tc_common.cuh", "device_utils.cuh", "sgemm_internal.h"]


SMALL_KERNEL_FILES = ["kernel_small.cu", "kernel_small.h", "sgemm_internal.h"]


SKINNY_KERNEL_FILES = ["kernel_skinny.cu", "kernel_presplit.cu", "kernel_tc_common.cuh", "device_utils.cuh",
                       "sgemm_internal.h"]


def tma_kernel_digest() -> str:
    """Hash of the sources of the TMA-fed FFMA kernel only (identifies the profiled kernel build)."""
    return _digest(TMA_KERNEL_FILES)


def tc_kernel_digest() -> str:
    """Hash of the sources of the 3xTF32 tensor-core kernel only."""
    return _digest(TC_KERNEL_FILES)


def pair_kernel_digest() -> str:
    """Hash of the sources of the CTA-pair tensor-core kernel only."""
    return _digest(PAIR_KERNEL_FILES)


def presplit_kernel_digest() -> str:
    """Hash of the sources of the split-operand kernels (split pass, GEMM, fixup) only."""
    return _digest(PRESPLIT_KERNEL_FILES)


def small_kernel_digest() -> str:
    """Hash of the sources of the small-product kernel only."""
    return _digest(SMALL_KERNEL_FILES)


def skinny_kernel_digest() -> str:
    """Hash of the sources of the short-side kernel and the split pass it runs first."""
    return _digest(SKINNY_KERNEL_FILES)


def _digest(files) -> str:
    h = hashlib.sha256()
    for name in files:
        h.update(name.encode())
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DIR, ("debug_" if debug else "") + os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DSGEMM_DEBUG_BOUNDS"] if debug else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libsgemm.so (debug=True: libsgemm_debug.so, the bounds-checking build) if
    any source changed; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    library = DEBUG_LIBRARY if debug else LIBRARY
    stamp = os.path.join(BUILD_DIR, "digest_debug.txt" if debug else "digest.txt")
    digest = source_digest()
    if not force and os.path.exists(library) and os.path.exists(stamp) and open(stamp).read() == digest:
        return library
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    tmp = library + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, library)
    with open(stamp, "w") as f:
        f.write(digest)
    return library


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
