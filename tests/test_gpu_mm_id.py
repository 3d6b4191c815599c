"""Routed experts (w4a16_mm_id) vs the oracle, plus bad ids and empty calls."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import EXPERTS, assert_parity, bf16_bits, sample_cols, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _experts(seed, E, N, K):
    hw = synth.make_weights(seed, N, K, E)
    return hw, ops.W4Matrix.from_host(hw)


@pytest.mark.parametrize("kernel", ["auto", "simt", "tc", "vanilla", "tc_stream", "tc_tile"])
def test_routed_experts_config(kernel):
    E, N, K = EXPERTS
    hw, w = _experts(0, E, N, K)
    T = 8
    ids_np = synth.make_ids(0, T, E)
    xb = synth.make_x(0, T, K)
    y = ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda(), kernel=kernel)
    cols = sample_cols(N, 2048)
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E, cols=cols,
                          threads=oracle.host_threads())
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"mm_id {kernel}")
    assert ops.device_status() == 0


@pytest.mark.parametrize("kernel", ["auto", "tc_stream"])
@pytest.mark.parametrize("T,E", [(1, 1), (3, 5), (20, 3), (64, 8)])
def test_routed_small_full(T, E, kernel):
    N, K = 70, 512
    hw, w = _experts(T * 10 + E, E, N, K)
    ids_np = synth.make_ids(T, T, E)
    xb = synth.make_x(E, T, K)
    y = ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda(), kernel=kernel)
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(y, yr, ad, f"mm_id T={T} E={E} {kernel}")


@pytest.mark.parametrize("kernel", ["tc_tile", "tc_stream"])
def test_bad_ids_tensor_core(kernel):
    """Out-of-range ids on the tensor-core launch shapes (K % 512 == 0), with
    several tiles per expert and an expert that takes two token chunks."""
    E, N, K = 5, 100, 1024
    hw, w = _experts(9, E, N, K)
    ids_np = np.array([1, -1, 3, 7, 1, 1, 0, 99, 1, 4, -5], dtype=np.int32)
    T = len(ids_np)
    xb = synth.make_x(9, T, K)
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda(), out=y, kernel=kernel)
    assert ops.device_status() & ops.DEVICE_BAD_ID
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(y, yr, ad, f"bad ids {kernel}")
    yb = bf16_bits(y)
    for t in (1, 3, 7, 10):
        assert np.all(yb[t] == 0)


def test_routed_launch_shapes_agree_bitwise():
    E, N, K, T = 6, 300, 2048, 37
    _, w = _experts(11, E, N, K)
    ids = torch.from_numpy(synth.make_ids(11, T, E)).cuda()
    x = to_dev_bf16(synth.make_x(11, T, K))
    a = bf16_bits(ops.mm_id(x, w, ids, kernel="tc_tile"))
    b = bf16_bits(ops.mm_id(x, w, ids, kernel="tc_stream"))
    assert np.array_equal(a, b)


def test_bad_ids_give_zero_rows_and_raise_the_flag():
    E, N, K, T = 4, 40, 128, 6
    hw, w = _experts(5, E, N, K)
    ids_np = np.array([1, -1, 3, 4, 0, 99], dtype=np.int32)
    xb = synth.make_x(5, T, K)
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda(), out=y)
    assert ops.device_status() & ops.DEVICE_BAD_ID
    assert ops.device_status() == 0  # reading clears it
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(y, yr, ad, "bad ids")
    yb = bf16_bits(y)
    for t in (1, 3, 5):
        assert np.all(yb[t] == 0)


def test_empty_token_list():
    E, N, K = 3, 32, 64
    _, w = _experts(6, E, N, K)
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, dtype=torch.int32, device="cuda")
    assert ops.mm_id(x, w, ids).shape == (0, N)


def test_all_tokens_on_one_expert_spans_chunks():
    E, N, K, T = 4, 96, 1024, 19
    hw, w = _experts(7, E, N, K)
    ids_np = np.full(T, 2, dtype=np.int32)
    xb = synth.make_x(7, T, K)
    y = ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda())
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(y, yr, ad, "one expert, 19 tokens")


@pytest.mark.parametrize("kernel", ["auto", "tc_stream", "tc_tile"])
def test_routed_rows_equal_mm_on_the_expert(kernel):
    """Every routed row is the w4a16_mm result of its token on the selected
    expert, bit for bit (the same canonical arithmetic on every launch shape)."""
    E, N, K = EXPERTS
    _, w = _experts(0, E, N, K)
    T = 8
    ids_np = synth.make_ids(0, T, E)
    x = to_dev_bf16(synth.make_x(0, T, K))
    y = bf16_bits(ops.mm_id(x, w, torch.from_numpy(ids_np).cuda(), kernel=kernel))
    for t in range(T):
        e = int(ids_np[t])
        we = ops.W4Matrix(w.Wq[e], w.scales[e], w.biases[e], N, K)
        assert np.array_equal(y[t], bf16_bits(ops.mm(x[t:t + 1], we, kernel="tc"))[0]), f"token {t}"


def test_routed_many_tokens_take_the_other_launch_shapes():
    """More tokens than the persistent routed mode takes (64): the tile and
    per-expert kernels, still equal to each other bit for bit."""
    E, N, K, T = 3, 200, 1024, 80
    hw, w = _experts(12, E, N, K)
    ids_np = synth.make_ids(12, T, E)
    ids = torch.from_numpy(ids_np).cuda()
    xb = synth.make_x(12, T, K)
    x = to_dev_bf16(xb)
    a = ops.mm_id(x, w, ids, kernel="tc_stream")
    b = ops.mm_id(x, w, ids)
    assert np.array_equal(bf16_bits(a), bf16_bits(b))
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(a, yr, ad, "mm_id T=80")


@pytest.mark.parametrize("T,E,same", [(32, 40, False), (32, 3, True), (31, 9, False), (2, 2, True)])
def test_routed_persistent_mode_edges(T, E, same):
    """The persistent routed mode at its token limit (32), with more experts
    than tokens, one expert taking every token (four chunks of eight), a row
    count that is not a multiple of the 32-row unit, and K = 1536 (three
    slice sums folded per unit); bitwise equal to the tile launch shape."""
    N, K = 200, 1536
    hw, w = _experts(T + 100 * E, E, N, K)
    ids_np = np.full(T, E - 1, dtype=np.int32) if same else synth.make_ids(T + E, T, E)
    ids = torch.from_numpy(ids_np).cuda()
    xb = synth.make_x(T * E, T, K)
    x = to_dev_bf16(xb)
    a = ops.mm_id(x, w, ids)
    b = ops.mm_id(x, w, ids, kernel="tc_tile")
    assert np.array_equal(bf16_bits(a), bf16_bits(b))
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(a, yr, ad, f"routed T={T} E={E}")
