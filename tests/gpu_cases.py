"""Shared builders for the GPU tests: seeded inputs, oracle references, checks.

Inputs come from the seeded generator (``skinny_gemm_gb300.synth``); expected
values come only from the CPU oracle (``oracle``).  The acceptance bound is
|y - y_ref| <= ulp_bf16(y_ref) + 1e-3 * sum_k |x w|, element by element.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from skinny_gemm_gb300 import ops, synth

# The workloads of the pages, named by what they are.
TINY = (256, 512)
DECODE_SET = {"q": (2048, 2560), "k": (512, 2560), "v": (512, 2560), "o": (2560, 2048),
              "gate": (10240, 2560), "up": (10240, 2560), "down": (2560, 10240)}
VERIFY_SHAPES = [(10240, 2560), (2560, 10240), (12288, 1536), (1536, 12288)]
LM_HEADS = [(262144, 1536), (262144, 2560)]
DENSE = (16384, 16384)
EXPERTS = (8, 6144, 2048)  # E, N, K


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


@functools.lru_cache(maxsize=8)
def host_weights(seed: int, N: int, K: int, E: int = 1) -> synth.HostW4:
    return synth.make_weights(seed, N, K, E)


_dev_cache: dict = {}


def dev_weights(seed: int, N: int, K: int, E: int = 1) -> ops.W4Matrix:
    key = (seed, N, K, E)
    if key not in _dev_cache:
        if len(_dev_cache) >= 4:
            _dev_cache.pop(next(iter(_dev_cache)))
        _dev_cache[key] = ops.W4Matrix.from_host(host_weights(seed, N, K, E))
    return _dev_cache[key]


def oracle_mm(x_bits: np.ndarray, hw: synth.HostW4, cols=None):
    M = x_bits.shape[0]
    return oracle.mm(x_bits, hw.Wq, hw.scales, hw.biases, M, hw.N, hw.K, cols=cols, threads=oracle.host_threads())


def assert_parity(y_dev: torch.Tensor, y_ref: np.ndarray, absdot: np.ndarray, what: str = "") -> float:
    """Element-wise acceptance; returns the worst |err| / bound ratio."""
    y = bf16_f64(y_dev).reshape(y_ref.shape)
    bound = oracle.tolerance(y_ref, absdot)
    err = np.abs(y - y_ref)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    ratio = err / bound
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    assert np.all(err <= bound), (f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance; worst at "
                                  f"{worst}: y={y[worst]!r} ref={y_ref[worst]!r} bound={bound[worst]:.3e}")
    return float(ratio.max())


def sample_cols(N: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last, and n random output columns (sorted, unique)."""
    rng = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, size=n)]))
    return cols.astype(np.int64)
