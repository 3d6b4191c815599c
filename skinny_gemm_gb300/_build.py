"""In-tree build of the native libraries (no cmake, no setuptools).

* ``lib/libw4a16.so``        -- the CUDA kernels and the C-ABI (``include/w4a16.h``),
                                compiled for sm_103a only.
* ``lib/libw4a16_synth.so``  -- the seeded input generator (``include/w4a16_synth.h``).

Each CUDA translation unit is compiled in parallel, then linked once.  A
library is rebuilt only when a source or header is newer than it.  The CUDA
runtime is linked statically and the driver API is reached through
``cudaGetDriverEntryPoint``, so the library loads on a host without a GPU
driver (its compute calls then fail with an error status).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
BUILDDIR = os.path.join(PKG, "_build")

CUDA_LIB = os.path.join(LIBDIR, "libw4a16.so")
SYNTH_LIB = os.path.join(LIBDIR, "libw4a16_synth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: only the explicit fused multiply-adds in the source are fused,
# so every instantiation of a kernel rounds in exactly the written order.
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC]
CC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a16.so")


def _newest(paths) -> float:
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def _stale(out: str, deps) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < _newest(deps)


def _run(cmd) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build_synth(force: bool = False) -> str:
    src = os.path.join(CSRC, "synth.c")
    deps = [src, os.path.join(INCLUDE, "w4a16_synth.h")]
    with _lock:
        if force or _stale(SYNTH_LIB, deps):
            os.makedirs(LIBDIR, exist_ok=True)
            tmp = SYNTH_LIB + f".tmp{os.getpid()}"
            _run(["gcc", *CC_FLAGS, "-I", INCLUDE, src, "-o", tmp, "-lm"])
            os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def cuda_sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build_cuda(force: bool = False, jobs: int | None = None, extra_flags: list[str] | None = None) -> str:
    srcs = cuda_sources()
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    with _lock:
        if not force and not _stale(CUDA_LIB, srcs + headers + [__file__]):
            return CUDA_LIB
        nvcc = _nvcc()
        os.makedirs(BUILDDIR, exist_ok=True)
        os.makedirs(LIBDIR, exist_ok=True)
        flags = NVCC_FLAGS + (extra_flags or [])

        def compile_one(src: str) -> str:
            obj = os.path.join(BUILDDIR, os.path.basename(src) + ".o")
            _run([nvcc, *flags, "-c", src, "-o", obj])
            return obj

        with ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp = CUDA_LIB + f".tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp])
        os.replace(tmp, CUDA_LIB)
    return CUDA_LIB


def build_all(force: bool = False) -> tuple[str, str]:
    with ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build_cuda, force)
        b = ex.submit(build_synth, force)
        return a.result(), b.result()
