"""Bit-exact debug entry points: w4a16_unpack and w4a16_dequant vs the oracle
(tiny-llm "Week 2 Day 2: Keep W4 Packed", sections "Packed Storage Layout"
and "Reconstruct a Stored Group")."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import host_weights, dev_weights, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(1, 64), (37, 192), (256, 512), (2048, 2560)])
def test_unpack_bit_exact(N, K):
    hw = host_weights(40, N, K)
    q = ops.unpack(dev_weights(40, N, K)).cpu().numpy()
    assert np.array_equal(q, oracle.unpack(hw.Wq, N, K))


@pytest.mark.parametrize("N,K", [(1, 64), (37, 192), (256, 512), (2048, 2560)])
def test_dequant_bit_exact(N, K):
    hw = host_weights(41, N, K)
    w = ops.dequant(dev_weights(41, N, K)).cpu().numpy()
    ref = oracle.dequant(hw.Wq, hw.scales, hw.biases, N, K)
    # q*s + b is exact in fp64 here, so the single-rounding fp32 fma equals it rounded once
    assert np.array_equal(w, ref.astype(np.float32))


def test_dequant_signed_scales_and_page_endpoints():
    # scale = +-bf16(0.0867) with bias -0.5 / 0.8 (the page's worked example), all 16 codes
    N, K = 2, 64
    sb = int(oracle.bf16_from_f64(np.array([0.0867]))[0])
    s = np.array([[sb], [sb ^ 0x8000]], dtype=np.uint16)
    b = oracle.bf16_from_f64(np.array([[-0.5], [0.8]]))
    Wq = np.tile(np.array([0x76543210, 0xFEDCBA98] * 4, dtype=np.uint32), (2, 1))
    host = synth.HostW4(Wq, s, b, N, K)
    w = ops.dequant(ops.W4Matrix.from_host(host)).cpu().numpy()
    assert np.array_equal(w, oracle.dequant(Wq, s, b, N, K).astype(np.float32))
    assert w[0, 0] == -0.5 and abs(w[0, 15] - 0.8) < 0.01
    assert abs(w[1, 0] - 0.8) < 0.01 and abs(w[1, 15] + 0.5) < 0.01
