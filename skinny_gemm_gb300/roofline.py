"""Algorithmic byte and flop counts for the W4A16 path (the roofline numerators).

Byte model, tiny-llm "Week 2 Day 2: Keep W4 Packed", section "Revisit the
Decode Roofline": a packed weight costs half a byte of code plus its share of
one bf16 scale and one bf16 bias per group, i.e. ``0.5 + 4/G`` bytes
(0.53125 at G = 128, 0.5625 at G = 64).  One kernel launch must read every
weight byte once and the activations once, and write the outputs once:

    bytes(M, N, K) = N*K*(0.5 + 4/G) + 2*M*K + 2*M*N
    flops(M, N, K) = 2*M*N*K

For routed experts only the distinct experts that some token selects are
read; untouched experts cost nothing.
"""
from __future__ import annotations

GROUP = 64


def bytes_per_weight(group: int = GROUP) -> float:
    return 0.5 + 4.0 / group


def weight_bytes(N: int, K: int, group: int = GROUP) -> int:
    """Bytes of packed codes + scales + biases of an N x K matrix."""
    return N * K // 2 + 4 * N * (K // group)


def mm_bytes(M: int, N: int, K: int, group: int = GROUP) -> int:
    return weight_bytes(N, K, group) + 2 * M * K + 2 * M * N


def mm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def mm_id_bytes(ids, T: int, N: int, K: int, E: int, group: int = GROUP) -> tuple[int, int]:
    """(bytes, distinct experts touched) of a routed call."""
    touched = len({int(e) for e in ids[:T] if 0 <= int(e) < E})
    return touched * weight_bytes(N, K, group) + 2 * T * K + 2 * T * N, touched


# STQ1_0 ("Hy4-preview Metal kernels for llama.cpp", section "Notes and
# gotchas"): 42 bytes per 256 weights; float32 activations in, float32 out.
STQ1_BLOCK_WEIGHTS, STQ1_BLOCK_BYTES = 256, 42


def stq1_weight_bytes(N: int, K: int) -> int:
    return N * (K // STQ1_BLOCK_WEIGHTS) * STQ1_BLOCK_BYTES


def stq1_mm_bytes(M: int, N: int, K: int) -> int:
    return stq1_weight_bytes(N, K) + 4 * M * K + 4 * M * N


def stq1_mm_id_bytes(ids, T: int, N: int, K: int, E: int) -> tuple[int, int]:
    touched = len({int(e) for e in ids[:T] if 0 <= int(e) < E})
    return touched * stq1_weight_bytes(N, K) + 4 * T * K + 4 * T * N, touched
