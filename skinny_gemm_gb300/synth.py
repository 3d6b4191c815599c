"""Seeded synthetic inputs for the W4A16 path (host side, numpy arrays).

A thin ctypes layer over ``libw4a16_synth.so`` (source ``csrc/synth.c``,
definitions in ``include/w4a16_synth.h``).  It draws numbers and packs them;
it contains none of the quantized matmul's arithmetic, so both the CUDA path
and the CPU oracle can take their inputs from it.

bf16 arrays are returned as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import threading
from dataclasses import dataclass

import numpy as np

from . import _build

GROUP = 64

_lock = threading.Lock()
_lib = None


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build_synth()
            lib = ctypes.CDLL(path)
            P, u64, i64 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64
            lib.w4a16_synth_hash.argtypes = [u64, ctypes.c_uint32, u64, i64, P]
            lib.w4a16_synth_x.argtypes = [u64, u64, i64, P]
            lib.w4a16_synth_codes.argtypes = [u64, u64, i64, P]
            lib.w4a16_synth_group_params.argtypes = [u64, u64, i64, P, P]
            lib.w4a16_synth_ids.argtypes = [u64, i64, ctypes.c_int32, P]
            lib.w4a16_synth_x_f32.argtypes = [u64, u64, i64, P]
            lib.w4a16_synth_stq1.argtypes = [u64, u64, i64, P]
            lib.w4a16_synth_fp16.argtypes = [ctypes.c_float, P]
            for f in ("w4a16_synth_hash", "w4a16_synth_x", "w4a16_synth_codes",
                      "w4a16_synth_group_params", "w4a16_synth_ids", "w4a16_synth_threads",
                      "w4a16_synth_x_f32", "w4a16_synth_stq1", "w4a16_synth_fp16"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ok(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"w4a16 synth {what}: status {rc}")


def hashes(seed: int, tid: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _ok(_load().w4a16_synth_hash(seed, tid, offset, n, _p(out)), "hash")
    return out


def make_x(seed: int, M: int, K: int, row0: int = 0) -> np.ndarray:
    """Activations x[M][K] (bf16 bits), rows row0..row0+M-1 of the seeded stream."""
    out = np.empty((M, K), dtype=np.uint16)
    _ok(_load().w4a16_synth_x(seed, row0 * K, M * K, _p(out)), "x")
    return out


def make_codes(seed: int, N: int, K: int, E: int = 1) -> np.ndarray:
    """Packed codes Wq[N][K/8] (or [E][N][K/8] when E > 1), uint32."""
    shape = (N, K // 8) if E == 1 else (E, N, K // 8)
    out = np.empty(shape, dtype=np.uint32)
    _ok(_load().w4a16_synth_codes(seed, 0, out.size, _p(out)), "codes")
    return out


def make_group_params(seed: int, N: int, K: int, E: int = 1):
    """(scales, biases), each bf16 bits [N][K/64] (or [E][N][K/64])."""
    shape = (N, K // GROUP) if E == 1 else (E, N, K // GROUP)
    s = np.empty(shape, dtype=np.uint16)
    b = np.empty(shape, dtype=np.uint16)
    _ok(_load().w4a16_synth_group_params(seed, 0, s.size, _p(s), _p(b)), "group params")
    return s, b


def make_ids(seed: int, T: int, E: int) -> np.ndarray:
    out = np.empty(T, dtype=np.int32)
    _ok(_load().w4a16_synth_ids(seed, T, E, _p(out)), "ids")
    return out


@dataclass
class HostW4:
    """Packed W4A16 weights on the host: Wq u32 [.., N, K/8]; scales/biases bf16 bits [.., N, K/64]."""

    Wq: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    N: int
    K: int
    E: int = 1

    @property
    def nbytes(self) -> int:
        return self.Wq.nbytes + self.scales.nbytes + self.biases.nbytes


def make_weights(seed: int, N: int, K: int, E: int = 1) -> HostW4:
    """Seeded packed weights for an N x K matrix (E stacked experts when E > 1)."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    s, b = make_group_params(seed, N, K, E)
    return HostW4(make_codes(seed, N, K, E), s, b, N, K, E)


def make_x_f32(seed: int, M: int, K: int, row0: int = 0) -> np.ndarray:
    """Float32 activations x[M][K], rows row0..row0+M-1 of the seeded stream."""
    out = np.empty((M, K), dtype=np.float32)
    _ok(_load().w4a16_synth_x_f32(seed, row0 * K, M * K, _p(out)), "x f32")
    return out


STQ1_WEIGHTS = 256  # weights per STQ1_0 block
STQ1_BYTES = 42     # bytes per STQ1_0 block


def make_stq1(seed: int, N: int, K: int, E: int = 1) -> np.ndarray:
    """STQ1_0 blocks uint8 [N][K/256][42] (or [E][N][K/256][42]) in the page's layout."""
    if K % STQ1_WEIGHTS:
        raise ValueError("K must be a multiple of 256")
    shape = (N, K // STQ1_WEIGHTS, STQ1_BYTES) if E == 1 else (E, N, K // STQ1_WEIGHTS, STQ1_BYTES)
    out = np.empty(shape, dtype=np.uint8)
    _ok(_load().w4a16_synth_stq1(seed, 0, out.size // STQ1_BYTES, _p(out)), "stq1")
    return out


def fp16_bits(v: float) -> int:
    out = np.zeros(1, dtype=np.uint16)
    _ok(_load().w4a16_synth_fp16(ctypes.c_float(v), _p(out)), "fp16")
    return int(out[0])


def threads() -> int:
    return int(_load().w4a16_synth_threads())
