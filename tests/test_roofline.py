"""Byte model against the numbers the page prints.

tiny-llm "Week 2 Day 2: Keep W4 Packed", section "Revisit the Decode Roofline"
(fixture tests/golden/w2d2_roofline.txt).
"""
import os

import pytest

from skinny_gemm_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "w2d2_roofline.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_bytes_per_weight_matches_page():
    g = _golden()
    assert roofline.bytes_per_weight(int(g["group_size"])) == g["bytes_per_weight"]
    assert roofline.bytes_per_weight(64) == 0.5625


def test_streamed_bytes_and_intensity_match_page():
    g = _golden()
    n = int(g["projection_weights"])
    streamed = n * roofline.bytes_per_weight(int(g["group_size"]))
    assert round(streamed / 1e9, 3) == g["streamed_gb_per_token"]
    flops = 2 * n  # one multiply-add per weight at M = 1
    assert round(flops / 1e9, 3) == g["gflops_per_token"]
    assert round(flops / streamed, 3) == g["flops_per_byte"]


def test_weight_bytes_is_integer_model():
    # 16384 x 16384 at G = 64: 134,217,728 code bytes + 16,777,216 scale/bias bytes
    assert roofline.weight_bytes(16384, 16384) == 134217728 + 16777216
    assert roofline.mm_bytes(1, 256, 512) == 256 * 512 * 0.5625 + 2 * 512 + 2 * 256


def test_mm_id_counts_distinct_touched_experts():
    b, touched = roofline.mm_id_bytes([3, 0, 2, 4, 5, 4, 0, 6], 8, 6144, 2048, 8)
    assert touched == 6
    assert b == 6 * roofline.weight_bytes(6144, 2048) + 2 * 8 * 2048 + 2 * 8 * 6144
    b, touched = roofline.mm_id_bytes([-1, 9], 2, 64, 64, 8)
    assert touched == 0


def test_stq1_byte_model():
    """STQ1_0: 42 bytes per 256 weights ("Hy4-preview Metal kernels for
    llama.cpp", section "Notes and gotchas"), float32 activations and outputs."""
    assert roofline.stq1_weight_bytes(16384, 16384) == 16384 * 64 * 42
    assert roofline.stq1_mm_bytes(2, 6144, 2048) == 6144 * 8 * 42 + 4 * 2 * 2048 + 4 * 2 * 6144
    b, touched = roofline.stq1_mm_id_bytes([3, 0, 2, 4, 5, 4, 0, 6], 8, 6144, 2048, 8)
    assert touched == 6 and b == 6 * 6144 * 8 * 42 + 4 * 8 * 2048 + 4 * 8 * 6144


def test_bench_traffic_key_covers_the_dominant_kernel():
    """The ncu traffic of the bench line is keyed by the dominant kernel's
    sources: they exist, and a summary line for the kernel is on file."""
    import bench
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "skinny_gemm_gb300", "csrc")
    assert all(os.path.exists(os.path.join(csrc, f)) for f in bench.DOMINANT_SOURCES)
    assert len(bench.kernel_source_sha()) == 16
    t = bench.ncu_traffic(bench.DOMINANT_KERNEL)
    assert t is None or t > 0
    text = open(os.path.join(os.path.dirname(csrc), "..", "profiles", "traffic.txt")).read()
    assert any(line.split()[:1] == [bench.DOMINANT_KERNEL] for line in text.splitlines() if not line.startswith("#"))
