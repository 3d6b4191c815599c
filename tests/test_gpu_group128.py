"""Tables quantized with 128 codes per scale and bias (the tiny-llm book's
group size): parameters expanded once with w4a16_expand_groups, then the
group-64 kernels, against the oracle's group-128 definition."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_parity, bf16_bits, sample_cols, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def g128_weights(seed, N, K):
    """Seeded codes; one scale and bias per 128 codes (every other group-64
    draw of the generator, the same distributions)."""
    hw = synth.make_weights(seed, N, K)
    s = np.ascontiguousarray(hw.scales[:, ::2])
    b = np.ascontiguousarray(hw.biases[:, ::2])
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    wq = torch.from_numpy(hw.Wq.view(np.int32)).cuda()
    return hw.Wq, s, b, ops.W4Matrix.from_group(wq, dev(s), dev(b), N, K, 128)


def test_expand_is_a_repeat():
    N, K = 300, 1280
    s = synth.make_weights(1, N, K).scales[:, :K // 128].copy()
    src = torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).cuda()
    dst = torch.empty(N, K // 64, dtype=torch.bfloat16, device="cuda")
    assert ops.lib().w4a16_expand_groups(src.data_ptr(), dst.data_ptr(), N, K, 128, None) == ops.OK
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(dst), np.repeat(s, 2, axis=1))
    dst4 = torch.empty(N, K // 64, dtype=torch.bfloat16, device="cuda")
    s4 = np.ascontiguousarray(s[:, :K // 256])
    src4 = torch.from_numpy(s4.view(np.int16)).view(torch.bfloat16).cuda()
    assert ops.lib().w4a16_expand_groups(src4.data_ptr(), dst4.data_ptr(), N, K, 256, None) == ops.OK
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(dst4), np.repeat(s4, 4, axis=1))


@pytest.mark.parametrize("N,K,M", [(70, 1024, 1), (10240, 2560, 1), (2560, 10240, 5), (500, 384, 3), (333, 2048, 11)])
@pytest.mark.parametrize("kernel", [None, "tc_stream"])
def test_group128_parity(N, K, M, kernel):
    Wq, s, b, w = g128_weights(N + K, N, K)
    xb = synth.make_x(M + N, M, K)
    y = ops.mm(to_dev_bf16(xb), w, kernel=kernel)
    cols = sample_cols(N, 1024)
    yr, ad = oracle.mm(xb, Wq, s, b, M, N, K, cols=cols, threads=oracle.host_threads(), group=128)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"group 128 {N}x{K} M={M}")


def test_group128_lm_head_rows_invariant():
    N, K = 262144, 2560
    Wq, s, b, w = g128_weights(3, N, K)
    xb = synth.make_x(9, 3, K)
    x = to_dev_bf16(xb)
    y3 = bf16_bits(ops.mm(x, w))
    for m in range(3):
        assert np.array_equal(bf16_bits(ops.mm(x[m:m + 1], w))[0], y3[m])
    cols = sample_cols(N, 512)
    yr, ad = oracle.mm(xb, Wq, s, b, 3, N, K, cols=cols, threads=oracle.host_threads(), group=128)
    y = torch.from_numpy(y3.view(np.int16)).view(torch.bfloat16).cuda()
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, "group 128 LM head")


# ---- native group-128 reads (w4a16_mm_g): the tables as they are ------------------------

def g128_native(seed, N, K):
    """The same tables as g128_weights, as a native group-128 W4Matrix and as
    the group-64 expansion of them."""
    Wq, s, b, wexp = g128_weights(seed, N, K)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    wnat = ops.W4Matrix(wexp.Wq, dev(s), dev(b), N, K, group=128)
    return Wq, s, b, wnat, wexp


@pytest.mark.parametrize("N,K", [(1, 512), (31, 1024), (999, 1536), (1000, 2560), (4099, 4096), (96, 8192)])
@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_native_group128_parity_and_equal_to_expansion(N, K, M):
    """Against the oracle's group-128 definition element by element, and bit
    for bit against the group-64 kernels on the expanded tables.  Odd N with
    K / 64 bytes per parameter row leaves a parameter tail that is not a
    16-byte multiple (N = 999, 31, 1)."""
    Wq, s, b, wnat, wexp = g128_native(N + K + 5, N, K)
    xb = synth.make_x(M + 3, M, K)
    x = to_dev_bf16(xb)
    y = ops.mm(x, wnat)
    y_exp = ops.mm(x, wexp)
    y_nows = ops.mm(x, wnat, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_exp.view(torch.int16)), "native group 128 vs expanded tables"
    assert torch.equal(y.view(torch.int16), y_nows.view(torch.int16)), "with and without a workspace"
    yr, ad = oracle.mm(xb, Wq, s, b, M, N, K, threads=oracle.host_threads(), group=128)
    assert_parity(y, yr, ad, f"native group 128 {N}x{K} M={M}")
    assert ops.device_status() == 0


@pytest.mark.parametrize("N,K", [(262144, 2560), (262144, 1536), (12288, 8192)])
def test_native_group128_large_rows_invariant(N, K):
    """The LM heads and 12288x8192 (eight canonical K-slices, folded in order
    inside whole-K units): rows of an M = 3 call equal the M = 1 calls and
    the expanded tables' results; sampled columns against the oracle."""
    Wq, s, b, wnat, wexp = g128_native(7, N, K)
    xb = synth.make_x(10, 3, K)
    x = to_dev_bf16(xb)
    y3 = ops.mm(x, wnat)
    for m in range(3):
        assert torch.equal(ops.mm(x[m:m + 1], wnat).view(torch.int16), y3[m:m + 1].view(torch.int16))
    assert torch.equal(y3.view(torch.int16), ops.mm(x, wexp).view(torch.int16))
    cols = sample_cols(N, 384, seed=N + K)
    yr, ad = oracle.mm(xb, Wq, s, b, 3, N, K, cols=cols, threads=oracle.host_threads(), group=128)
    assert_parity(y3[:, torch.from_numpy(cols).cuda()], yr, ad, f"native group 128 {N}x{K}")


def test_native_group128_rejects():
    L = ops.lib()
    N, K = 64, 768  # K % 512 != 0: expand instead
    Wq, s, b, wnat, wexp = g128_native(1, 64, 1024)
    x = torch.zeros(1, 1024, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(1, 64, dtype=torch.bfloat16, device="cuda")
    args = (x.data_ptr(), wnat.Wq.data_ptr(), wnat.scales.data_ptr(), wnat.biases.data_ptr(), y.data_ptr())
    assert L.w4a16_mm_g(*args, 1, N, K, 128, None, 0, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_g(*args, 1, 64, 1024, 96, None, 0, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_g(*args, 1, 64, 1024 * 9, 128, None, 0, None) == ops.ERR_SHAPE
    with pytest.raises(ValueError):
        ops.mm(x, wnat, kernel="simt")
    with pytest.raises(ValueError):
        ops.mm_id(x, wnat, torch.zeros(1, dtype=torch.int32, device="cuda"))
