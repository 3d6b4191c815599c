"""w4a16_embed: quantized embedding rows, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import LM_HEADS, bf16_bits, dev_weights, host_weights
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,T", [(100, 64, 1), (1000, 192, 7), (333, 2560, 64), (5, 8192, 3)])
def test_rows_bit_exact(N, K, T):
    hw = synth.make_weights(N + K, N, K)
    w = ops.W4Matrix.from_host(hw)
    ids_np = synth.make_ids(T, T, N)
    out = ops.embed(torch.from_numpy(ids_np).cuda(), w)
    assert out.shape == (T, K)
    want = oracle.embed(hw.Wq, hw.scales, hw.biases, ids_np, N, K)
    assert np.array_equal(bf16_bits(out), want)
    assert ops.device_status() == 0


def test_vocabulary_table_repeated_and_bad_ids():
    """The 262144 x 2560 tied table; a repeated id, the first and last rows,
    ids out of range (zero rows and the device flag)."""
    N, K = LM_HEADS[1]
    hw = host_weights(1, N, K)
    ids_np = np.array([7, N - 1, 0, 7, -1, N, 123456], dtype=np.int32)
    out = torch.full((len(ids_np), K), 3.0, dtype=torch.bfloat16, device="cuda")
    ops.embed(torch.from_numpy(ids_np).cuda(), dev_weights(1, N, K), out=out)
    assert ops.device_status() & ops.DEVICE_BAD_ID
    got = bf16_bits(out)
    want = oracle.embed(hw.Wq, hw.scales, hw.biases, ids_np, N, K)
    assert np.array_equal(got, want)
    assert np.all(got[4] == 0) and np.all(got[5] == 0)


def test_rows_equal_dequant_rounded():
    """Each row is w4a16_dequant's fp32 row rounded to bf16 (the same single-
    rounding fma, then the output rounding)."""
    N, K = 64, 512
    hw = synth.make_weights(11, N, K)
    w = ops.W4Matrix.from_host(hw)
    full = ops.dequant(w)
    ids = torch.arange(N - 1, -1, -1, dtype=torch.int32, device="cuda")
    out = ops.embed(ids, w)
    assert torch.equal(out, full.flip(0).to(torch.bfloat16))


def test_empty():
    w = dev_weights(2, 10, 64)
    assert ops.embed(torch.empty(0, dtype=torch.int32, device="cuda"), w).shape == (0, 64)
