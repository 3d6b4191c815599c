"""w4a16_mm_argmax: the index and value of the largest output of every row.

The decision is taken on the kernel's own bf16 outputs (the precision the
kernel computes in): idx must equal the argmax of w4a16_mm's row bit for bit
(ties to the smallest index), and val the output there.  Against the oracle
the choice must be valid: the chosen output within tolerance of the oracle,
and no other output definitely larger (its oracle value above the chosen
one's by more than both tolerances).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import DENSE, LM_HEADS, bf16_bits, dev_weights, host_weights, oracle_mm, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def order_keys(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers in the order of their values (NaN above all)."""
    b = bits.astype(np.int64)
    nan = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    k = np.where(b & 0x8000, 0x7FFF - (b & 0x7FFF), 0x8000 + b)
    return np.where(nan, 0x10000, k)


def argmax_of(y_bits: np.ndarray) -> np.ndarray:
    return np.argmax(order_keys(y_bits), axis=-1)  # first maximum: the smallest index


def check(x_bits, w, hw, M, N, K, what, full_oracle=True):
    x = to_dev_bf16(x_bits)
    idx, val = ops.mm_argmax(x, w)
    y = bf16_bits(ops.mm(x, w, kernel="tc")).reshape(M, N)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
    want = argmax_of(y)
    got = idx.cpu().numpy()
    assert np.array_equal(got, want), f"{what}: argmax {got} != argmax of w4a16_mm {want}"
    assert np.array_equal(bf16_bits(val), y[np.arange(M), want]), f"{what}: values"
    # validity against the oracle: all columns, or the chosen one and the 64 largest outputs
    if full_oracle:
        cols = np.arange(N)
    else:
        top = np.argsort(-yf, axis=-1)[:, :64]
        cols = np.unique(np.concatenate([top.ravel(), got]))
    yr, ad = oracle_mm(x_bits, hw, cols=cols)
    tol = oracle.tolerance(yr, ad)
    pos = {c: i for i, c in enumerate(cols.tolist())}
    for m in range(M):
        j = pos[int(got[m])]
        assert abs(yf[m, got[m]] - yr[m, j]) <= tol[m, j], f"{what}: row {m} value outside tolerance"
        assert np.all(yr[m] <= yr[m, j] + tol[m] + tol[m, j]), f"{what}: row {m} has a definitely larger output"


@pytest.mark.parametrize("N,K,M", [(70, 512, 1), (1000, 1024, 3), (4097, 512, 8), (300, 2048, 11), (512, 16384, 2)])
def test_small_shapes_full_oracle(N, K, M):
    """Ragged row tiles, several chunks of rows (M = 11), and a K split into
    32 slices (512 x 16384: the reduction path)."""
    hw = host_weights(N + K, N, K)
    w = ops.W4Matrix.from_host(hw)
    check(synth.make_x(M, M, K), w, hw, M, N, K, f"{N}x{K} M={M}")


@pytest.mark.parametrize("N,K", LM_HEADS)
@pytest.mark.parametrize("M", [1, 3])
def test_lm_heads(N, K, M):
    hw = host_weights(1, N, K)
    check(synth.make_x(7 + M, M, K), dev_weights(1, N, K), hw, M, N, K, f"LM head {N}x{K} M={M}", full_oracle=False)


def test_dense_split_k():
    N, K = DENSE
    hw = host_weights(3, N, K)
    check(synth.make_x(4, 1, K), dev_weights(3, N, K), hw, 1, N, K, "16384^2", full_oracle=False)


def test_ties_go_to_the_smallest_index():
    """All-zero codes with one scale and bias everywhere: every output equal."""
    N, K = 5000, 1024
    hw = synth.make_weights(5, N, K)
    hw.Wq[:] = 0
    hw.scales[:] = hw.scales.flat[0]
    hw.biases[:] = hw.biases.flat[0]
    w = ops.W4Matrix.from_host(hw)
    x = to_dev_bf16(synth.make_x(5, 4, K))
    idx, val = ops.mm_argmax(x, w)
    assert np.all(idx.cpu().numpy() == 0)
    y = bf16_bits(ops.mm(x, w, kernel="tc"))
    assert np.all(y == y[:, :1]) and np.array_equal(bf16_bits(val), y[:, 0])


def test_nan_output_ranks_first():
    N, K = 3000, 512
    hw = synth.make_weights(6, N, K)
    hw.scales[1234, 3] = 0x7FC0  # NaN scale: output row 1234 is NaN
    hw.scales[2900, 0] = 0x7FC0
    w = ops.W4Matrix.from_host(hw)
    idx, val = ops.mm_argmax(to_dev_bf16(synth.make_x(6, 2, K)), w)
    assert np.all(idx.cpu().numpy() == 1234)
    v = bf16_bits(val)
    assert np.all(((v & 0x7F80) == 0x7F80) & ((v & 0x7F) != 0))


def test_without_values_and_interleaved_with_mm():
    """val = None; calls on one stream with w4a16_mm in between (the shared
    workspace is left clean by every launch); eager and in a CUDA graph."""
    N, K = 20000, 1536
    hw = host_weights(8, N, K)
    w = ops.W4Matrix.from_host(hw)
    xs = [to_dev_bf16(synth.make_x(20 + i, 2, K)) for i in range(3)]
    want = [argmax_of(bf16_bits(ops.mm(x, w, kernel="tc"))) for x in xs]
    for i, x in enumerate(xs):
        idx, val = ops.mm_argmax(x, w, val=False)
        assert val is None and np.array_equal(idx.cpu().numpy(), want[i])
        ops.mm(x, w)
    outs = [torch.empty(2, dtype=torch.int32, device="cuda") for _ in xs]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ops.mm_argmax(xs[0], w, idx=outs[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, o in zip(xs, outs):
            ops.mm_argmax(x, w, idx=o)
            ops.mm(x, w)
    for _ in range(3):
        for o in outs:
            o.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        for o, wv in zip(outs, want):
            assert np.array_equal(o.cpu().numpy(), wv)


def test_rejects_other_k():
    w = dev_weights(9, 64, 448)
    with pytest.raises(ValueError):
        ops.mm_argmax(to_dev_bf16(synth.make_x(9, 1, 448)), w)
