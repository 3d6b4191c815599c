"""CPU oracle for the W4A16 group-affine quantized matmul -- TEST INFRASTRUCTURE.

Only ``tests/``, the package smoke check in ``__graft_entry__`` and the
``cpu_baseline`` / reference leg of ``bench.py`` load this module.  The product
path never imports it and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (plain C++17, fp64, multithreaded over
output columns).  This file only builds that library and marshals numpy
arrays into it.  bf16 tensors are passed as ``numpy.uint16`` bit patterns.

Citations (page titles; sections in quotes):
  [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
  [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
         speculative decoding" (RESMP-DEV model card)

Acceptance bound used by the parity tests (written out in ``tolerance``):
  |y - y_ref| <= ulp_bf16(y_ref) + 1e-3 * sum_k |x[m,k] * w[n,k]|
and for the float32 STQ1_0 path of [HY4] ``stq1_tolerance``.

  [HY4]  "Hy4-preview Metal kernels for llama.cpp"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_w4a16.so")
_lock = threading.Lock()
_lib = None

GROUP = 64

# Portable flags: no SIMD intrinsics, no -march, and no fused multiply-add
# contraction so x86 and arm64 hosts round identically.
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB, extra: list[str] | None = None, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out`` (skipped when up to date)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", *CXXFLAGS, *(extra or []), src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int
    lib.oracle_group_size.restype = i32
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_bf16_from_double_array.argtypes = [P, i64, P, i32]
    lib.oracle_bf16_from_double_array.restype = None
    lib.oracle_bf16_from_float_array.argtypes = [P, i64, P, i32]
    lib.oracle_bf16_from_float_array.restype = None
    lib.oracle_ulp_bf16.argtypes = [ctypes.c_double]
    lib.oracle_ulp_bf16.restype = ctypes.c_double
    lib.oracle_bf16_to_double_array.argtypes = [P, i64, P]
    lib.oracle_bf16_to_double_array.restype = None
    lib.oracle_ulp_bf16_array.argtypes = [P, i64, P]
    lib.oracle_ulp_bf16_array.restype = None
    lib.oracle_unpack.argtypes = [P, i64, i64, P]
    lib.oracle_unpack.restype = i32
    lib.oracle_dequant.argtypes = [P, P, P, i64, i64, P]
    lib.oracle_dequant.restype = i32
    lib.oracle_dequant_g.argtypes = [P, P, P, i64, i64, i64, P]
    lib.oracle_dequant_g.restype = i32
    lib.oracle_mm.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P, P, i32]
    lib.oracle_mm.restype = i32
    lib.oracle_mm_g.argtypes = [P, P, P, P, i64, i64, i64, i64, P, i64, P, P, i32]
    lib.oracle_mm_g.restype = i32
    lib.oracle_mm_id.argtypes = [P, P, P, P, P, i64, i64, i64, i64, P, i64, P, P, i32]
    lib.oracle_mm_id.restype = i32
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = ctypes.c_double
    lib.oracle_stq1_lanes.argtypes = [i32, i32, P]
    lib.oracle_stq1_lanes.restype = i32
    lib.oracle_stq1_dequant.argtypes = [P, i64, i64, P]
    lib.oracle_stq1_dequant.restype = i32
    lib.oracle_stq1_mm.argtypes = [P, P, i64, i64, i64, P, i64, P, P, i32]
    lib.oracle_stq1_mm.restype = i32
    lib.oracle_stq1_mm_id.argtypes = [P, P, P, i64, i64, i64, i64, P, i64, P, P, i32]
    lib.oracle_stq1_mm_id.restype = i32
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


class Oracle:
    """The oracle library behind numpy marshalling (one per loaded .so)."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    # -- bf16, written in oracle.cpp from the format definition --
    def bf16_to_f64(self, bits) -> np.ndarray:
        b = _c(bits, np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_bf16_to_double_array(_ptr(b), b.size, _ptr(out))
        return out

    def bf16_from_f64(self, v, threads: int = 0) -> np.ndarray:
        a = _c(v, np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_bf16_from_double_array(_ptr(a), a.size, _ptr(out), threads)
        return out

    def bf16_from_f32(self, v, threads: int = 0) -> np.ndarray:
        a = _c(v, np.float32)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_bf16_from_float_array(_ptr(a), a.size, _ptr(out), threads)
        return out

    def ulp_bf16(self, v) -> np.ndarray:
        a = _c(v, np.float64)
        out = np.empty(a.shape, dtype=np.float64)
        self.lib.oracle_ulp_bf16_array(_ptr(a), a.size, _ptr(out))
        return out

    def tolerance(self, y_ref: np.ndarray, absdot: np.ndarray) -> np.ndarray:
        """Per-element acceptance bound: ulp_bf16(y_ref) + 1e-3 * sum_k |x w|."""
        return self.ulp_bf16(y_ref) + 1e-3 * np.asarray(absdot, dtype=np.float64)

    # -- the definition --
    def unpack(self, Wq: np.ndarray, N: int, K: int) -> np.ndarray:
        """Codes q[N][K] (uint8) from packed Wq[N][K/8]."""
        w = _c(Wq, np.uint32)
        q = np.empty((N, K), dtype=np.uint8)
        _check(self.lib.oracle_unpack(_ptr(w), N, K, _ptr(q)), "unpack")
        return q

    def dequant(self, Wq, scales, biases, N: int, K: int, group: int = GROUP) -> np.ndarray:
        """Weights w[N][K] = q*s + b in fp64 (scale and bias per `group` codes)."""
        w_ = _c(Wq, np.uint32)
        s, b = _c(scales, np.uint16), _c(biases, np.uint16)
        out = np.empty((N, K), dtype=np.float64)
        if group == GROUP:
            rc = self.lib.oracle_dequant(_ptr(w_), _ptr(s), _ptr(b), N, K, _ptr(out))
        else:
            rc = self.lib.oracle_dequant_g(_ptr(w_), _ptr(s), _ptr(b), N, K, group, _ptr(out))
        _check(rc, "dequant")
        return out

    def embed(self, Wq, scales, biases, ids, N: int, K: int) -> np.ndarray:
        """bf16 bits [T][K] of the table rows ids ([W2D2] "Task 1: Implement
        Quantized Linear and Embedding": row lookup, unpack, q * scale +
        bias): the exact q*s + b of ``dequant``, rounded once to fp32 (what a
        single-rounding fma gives) and then to bf16 with ``bf16_from_f32``.
        An id outside 0..N-1 gives a row of zeros."""
        ids = np.asarray(ids, dtype=np.int64).reshape(-1)
        ok = (ids >= 0) & (ids < N)
        rows = np.where(ok, ids, 0)
        Wq = np.asarray(Wq).reshape(N, K // 8)
        s = np.asarray(scales).reshape(N, K // GROUP)
        b = np.asarray(biases).reshape(N, K // GROUP)
        w = self.dequant(Wq[rows], s[rows], b[rows], len(ids), K)
        out = self.bf16_from_f32(w.astype(np.float32)).reshape(len(ids), K)
        out[~ok] = 0
        return out

    def mm(self, x, Wq, scales, biases, M: int, N: int, K: int, cols=None, threads: int = 0, group: int = GROUP):
        """(y, absdot), both fp64 [M][ncols]: y = x W^T on the sampled columns
        (scale and bias per `group` codes: 64, or the book's 128)."""
        x_ = _c(x, np.uint16)
        w_ = _c(Wq, np.uint32)
        s, b = _c(scales, np.uint16), _c(biases, np.uint16)
        c = None if cols is None else _c(cols, np.int64)
        nc = N if c is None else c.size
        y = np.empty((M, nc), dtype=np.float64)
        ad = np.empty((M, nc), dtype=np.float64)
        if group == GROUP:
            rc = self.lib.oracle_mm(_ptr(x_), _ptr(w_), _ptr(s), _ptr(b), M, N, K, _ptr(c), nc, _ptr(y), _ptr(ad),
                                    threads)
        else:
            rc = self.lib.oracle_mm_g(_ptr(x_), _ptr(w_), _ptr(s), _ptr(b), M, N, K, group, _ptr(c), nc, _ptr(y),
                                      _ptr(ad), threads)
        _check(rc, "mm")
        return y, ad

    def mm_id(self, x, Wq, scales, biases, ids, T: int, N: int, K: int, E: int, cols=None, threads: int = 0):
        """(y, absdot), fp64 [T][ncols]: y[t] = W[ids[t]] x[t]; bad ids give zero rows."""
        x_ = _c(x, np.uint16)
        w_ = _c(Wq, np.uint32)
        s, b = _c(scales, np.uint16), _c(biases, np.uint16)
        i_ = _c(ids, np.int32)
        c = None if cols is None else _c(cols, np.int64)
        nc = N if c is None else c.size
        y = np.empty((T, nc), dtype=np.float64)
        ad = np.empty((T, nc), dtype=np.float64)
        _check(self.lib.oracle_mm_id(_ptr(x_), _ptr(w_), _ptr(s), _ptr(b), _ptr(i_), T, N, K, E, _ptr(c), nc,
                                     _ptr(y), _ptr(ad), threads), "mm_id")
        return y, ad

    # -- STQ1_0, the ternary format of [HY4] (blocks: uint8 [N][K/256][42]) --
    def fp16_to_f64(self, h: int) -> float:
        return self.lib.oracle_fp16_to_double(int(h) & 0xFFFF)

    def stq1_lanes(self, c: int, s: int) -> list[int]:
        """The four lane values of group code c under group sign bit s."""
        v = np.zeros(4, dtype=np.int32)
        _check(self.lib.oracle_stq1_lanes(int(c), int(s), _ptr(v)), "stq1_lanes")
        return [int(t) for t in v]

    def stq1_dequant(self, blocks, N: int, K: int) -> np.ndarray:
        """Weights w[N][K] = d * v in fp64."""
        b = _c(blocks, np.uint8)
        out = np.empty((N, K), dtype=np.float64)
        _check(self.lib.oracle_stq1_dequant(_ptr(b), N, K, _ptr(out)), "stq1_dequant")
        return out

    def stq1_mm(self, x, blocks, M: int, N: int, K: int, cols=None, threads: int = 0):
        """(y, absdot), fp64 [M][ncols]: y = x W^T for float32 x [M][K]."""
        x_ = _c(x, np.float32)
        b = _c(blocks, np.uint8)
        c = None if cols is None else _c(cols, np.int64)
        nc = N if c is None else c.size
        y = np.empty((M, nc), dtype=np.float64)
        ad = np.empty((M, nc), dtype=np.float64)
        _check(self.lib.oracle_stq1_mm(_ptr(x_), _ptr(b), M, N, K, _ptr(c), nc, _ptr(y), _ptr(ad), threads),
               "stq1_mm")
        return y, ad

    def stq1_mm_id(self, x, blocks, ids, T: int, N: int, K: int, E: int, cols=None, threads: int = 0):
        """(y, absdot), fp64 [T][ncols]: y[t] = W[ids[t]] x[t]; bad ids give zero rows."""
        x_ = _c(x, np.float32)
        b = _c(blocks, np.uint8)
        i_ = _c(ids, np.int32)
        c = None if cols is None else _c(cols, np.int64)
        nc = N if c is None else c.size
        y = np.empty((T, nc), dtype=np.float64)
        ad = np.empty((T, nc), dtype=np.float64)
        _check(self.lib.oracle_stq1_mm_id(_ptr(x_), _ptr(b), _ptr(i_), T, N, K, E, _ptr(c), nc, _ptr(y), _ptr(ad),
                                          threads), "stq1_mm_id")
        return y, ad

    def stq1_get_rows(self, blocks, ids, N: int, K: int) -> np.ndarray:
        """float32 [T][K]: the weights d * v of the rows ids ([HY4] kernel table:
        kernel_get_rows_stq1_0, the row gather), exact in float32; an id outside
        0..N-1 gives a row of zeros."""
        ids = np.asarray(ids, dtype=np.int64).reshape(-1)
        ok = (ids >= 0) & (ids < N)
        b = np.asarray(blocks, dtype=np.uint8).reshape(N, -1)
        w = self.stq1_dequant(b[np.where(ok, ids, 0)], len(ids), K)
        out = w.astype(np.float32)
        out[~ok] = 0
        return out


def stq1_tolerance(absdot, K: int) -> np.ndarray:
    """Acceptance bound for the float32 STQ1_0 outputs:
        |y - y_ref| <= (2^-16 + (K/256 + 16) * 2^-23) * sum_k |x[m,k] * w[n,k]|
    The activations enter the tensor cores as three bf16 parts that sum to x
    exactly; the products with ternary weights are exact; what rounds is the
    fp32 accumulation: 16 steps of 16 products per 256-weight block (each
    step allowed a 2^-22 relative error), then one fused multiply-add with
    the block scale per block, the K-slice sums and the sum of the three
    parts (one 2^-24 rounding each, bounded here by 2^-23 apiece)."""
    return (2.0 ** -16 + (K // 256 + 16) * 2.0 ** -23) * np.asarray(absdot, dtype=np.float64)


_default = None


def default() -> Oracle:
    """The oracle built from ``oracle.cpp`` in this directory."""
    global _default
    if _default is None:
        _default = Oracle(load())
    return _default


def bf16_to_f64(bits):
    return default().bf16_to_f64(bits)


def bf16_from_f64(v, threads: int = 0):
    return default().bf16_from_f64(v, threads)


def bf16_from_f32(v, threads: int = 0):
    return default().bf16_from_f32(v, threads)


def ulp_bf16(v):
    return default().ulp_bf16(v)


def tolerance(y_ref, absdot):
    return default().tolerance(y_ref, absdot)


def unpack(Wq, N, K):
    return default().unpack(Wq, N, K)


def dequant(Wq, scales, biases, N, K, group: int = GROUP):
    return default().dequant(Wq, scales, biases, N, K, group)


def embed(Wq, scales, biases, ids, N, K):
    return default().embed(Wq, scales, biases, ids, N, K)


def mm(x, Wq, scales, biases, M, N, K, cols=None, threads: int = 0, group: int = GROUP):
    return default().mm(x, Wq, scales, biases, M, N, K, cols, threads, group)


def mm_id(x, Wq, scales, biases, ids, T, N, K, E, cols=None, threads: int = 0):
    return default().mm_id(x, Wq, scales, biases, ids, T, N, K, E, cols, threads)


def stq1_dequant(blocks, N, K):
    return default().stq1_dequant(blocks, N, K)


def stq1_mm(x, blocks, M, N, K, cols=None, threads: int = 0):
    return default().stq1_mm(x, blocks, M, N, K, cols, threads)


def stq1_mm_id(x, blocks, ids, T, N, K, E, cols=None, threads: int = 0):
    return default().stq1_mm_id(x, blocks, ids, T, N, K, E, cols, threads)


def stq1_get_rows(blocks, ids, N, K):
    return default().stq1_get_rows(blocks, ids, N, K)


def host_threads() -> int:
    """Cores this process may run on (the affinity mask), used as the thread count."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)
