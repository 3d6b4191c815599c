"""The tcgen05 prefill kernel (the default above 32 rows, any M when selected):
parity with the oracle, and the rows' relation to M = 1 calls.

Each 64-code group of a 128-row weight tile is expanded once to bf16 in
shared memory and multiplied with up to 128 activation rows by tcgen05.mma
into tensor memory; the per-group rescale and the slice sums follow the
canonical arithmetic of the skinny kernels.
"""
import numpy as np
import pytest
import torch

from gpu_cases import assert_parity, dev_weights, host_weights, oracle_mm, sample_cols, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("N,K", [(1, 512), (127, 512), (300, 1024), (1000, 2048), (2560, 1536)])
@pytest.mark.parametrize("M", [16, 17, 33, 64, 100, 128, 129, 200])
def test_prefill_parity_ragged(N, K, M):
    hw = host_weights(N + K, N, K)
    w = dev_weights(N + K, N, K)
    xb = synth.make_x(M + 7, M, K)
    y = ops.mm(to_dev_bf16(xb), w, kernel="tc_prefill")
    torch.cuda.synchronize()
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"prefill M={M} N={N} K={K}")
    assert ops.device_status() == 0


@pytest.mark.parametrize("N,K", [(10240, 2560), (12288, 1536), (2560, 10240)])
@pytest.mark.parametrize("M", [16, 32, 64, 128])
def test_prefill_parity_layer_shapes(N, K, M):
    """The verify/prefill projection shapes (several canonical K-slices on
    2560x10240), sampled output columns against the oracle."""
    hw = host_weights(3, N, K)
    w = dev_weights(3, N, K)
    xb = synth.make_x(M + 11, M, K)
    y = ops.mm(to_dev_bf16(xb), w, kernel="tc_prefill")
    cols = sample_cols(N, 384, seed=M)
    yr, ad = oracle_mm(xb, hw, cols)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"prefill M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(300, 1024), (10240, 2560), (2560, 10240)])
def test_prefill_rows_equal_single_row_calls(N, K):
    """Each row of a many-row call against the skinny kernels' M = 1 call on
    that row: both take the same canonical sums (the same sixteen codes per
    MMA step, the same group rescale and slice order)."""
    w = dev_weights(4, N, K)
    M = 40
    xb = synth.make_x(13, M, K)
    x = to_dev_bf16(xb)
    y = ops.mm(x, w)  # M > 32: the prefill kernel by default
    assert torch.equal(_bits(y), _bits(ops.mm(x, w, kernel="tc_prefill")))
    rows = [0, 1, 17, 31, 32, 39]
    ones = torch.stack([ops.mm(x[m:m + 1], w)[0] for m in rows])
    torch.cuda.synchronize()
    got = y[rows]
    same = (_bits(got) == _bits(ones)).float().mean().item()
    assert same == 1.0, f"{100 * (1 - same):.3f}% of the row outputs differ from M = 1 calls"


def test_prefill_selected_for_few_rows_and_dense():
    """The kernel selected explicitly at M = 1..8 equals its own many-row
    results row by row, and the 16384^2 matrix at M = 16 passes parity."""
    N, K = 1000, 2048
    w = dev_weights(5, N, K)
    xb = synth.make_x(21, 24, K)
    x = to_dev_bf16(xb)
    y = ops.mm(x, w, kernel="tc_prefill")
    for M in (1, 3, 8):
        assert torch.equal(_bits(ops.mm(x[:M], w, kernel="tc_prefill")), _bits(y[:M]))
    N, K = 16384, 16384
    xb = synth.make_x(22, 16, K)
    y = ops.mm(to_dev_bf16(xb), dev_weights(6, N, K), kernel="tc_prefill")
    cols = sample_cols(N, 128, seed=6)
    yr, ad = oracle_mm(xb, host_weights(6, N, K), cols)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, "prefill 16384^2 M=16")
    assert ops.device_status() == 0
