"""w4a16_mm_group: independent projections that share K and M in one launch.
Every item must equal w4a16_mm on it bit for bit (and hence the oracle
within the tolerance), whether the group runs as one launch or falls back
to consecutive calls."""
import numpy as np
import pytest
import torch

from gpu_cases import assert_parity, bf16_bits, dev_weights, host_weights, oracle_mm, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

GROUPS = {
    "qkv": [(2048, 2560), (512, 2560), (512, 2560)],
    "gate_up": [(10240, 2560), (10240, 2560)],
    "ragged": [(1, 512), (33, 512), (1000, 512), (17, 512)],
    "deep_k": [(300, 10240), (2560, 10240)],
    "eight": [(16 * i + 5, 1024) for i in range(8)],
    "tail_k": [(64, 768), (96, 768), (300, 768)],
    "too_large_fallback": [(20000, 4096), (64, 4096)],
}


@pytest.mark.parametrize("name", sorted(GROUPS))
@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_group_equals_separate_calls(name, M):
    shapes = GROUPS[name]
    ws = [dev_weights(50 + i, N, K) for i, (N, K) in enumerate(shapes)]
    xs = [to_dev_bf16(synth.make_x(60 + i, M, K)) for i, (N, K) in enumerate(shapes)]
    ys = ops.mm_group(xs, ws)
    for i, (x, w, y) in enumerate(zip(xs, ws, ys)):
        ref = ops.mm(x, w)
        assert np.array_equal(bf16_bits(y), bf16_bits(ref)), f"{name} item {i} M={M}"


def test_group_matches_oracle():
    shapes = GROUPS["ragged"]
    M = 5
    xbs = [synth.make_x(70 + i, M, K) for i, (N, K) in enumerate(shapes)]
    ws = [dev_weights(80 + i, N, K) for i, (N, K) in enumerate(shapes)]
    ys = ops.mm_group([to_dev_bf16(xb) for xb in xbs], ws)
    for i, ((N, K), xb, y) in enumerate(zip(shapes, xbs, ys)):
        yr, ad = oracle_mm(xb, host_weights(80 + i, N, K))
        assert_parity(y, yr, ad, f"group item {i}")


def test_group_writes_only_its_outputs():
    shapes = GROUPS["qkv"]
    ws = [dev_weights(90 + i, N, K) for i, (N, K) in enumerate(shapes)]
    xs = [to_dev_bf16(synth.make_x(91 + i, 1, K)) for i, (N, K) in enumerate(shapes)]
    flat = torch.full((sum(N for N, _ in shapes) + 64,), 5.0, dtype=torch.bfloat16, device="cuda")
    outs, off = [], 32
    for N, _ in shapes:
        outs.append(flat[off:off + N].view(1, N))  # contiguous views into one buffer
        off += N
    ops.mm_group(xs, ws, outs)
    for y, x, w in zip(outs, xs, ws):
        assert np.array_equal(bf16_bits(y), bf16_bits(ops.mm(x, w)))
    assert torch.all(flat[:32] == 5.0) and torch.all(flat[off:] == 5.0)


def test_group_rejects_mixed_k():
    ws = [dev_weights(95, 64, 512), dev_weights(96, 64, 1024)]
    xs = [torch.zeros(1, 512, dtype=torch.bfloat16, device="cuda"), torch.zeros(1, 1024, dtype=torch.bfloat16,
                                                                              device="cuda")]
    with pytest.raises(ValueError):
        ops.mm_group(xs, ws)
