"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import (DECODE_SET, DENSE, LM_HEADS, TINY, VERIFY_SHAPES, assert_parity, bf16_bits, dev_weights,
                       host_weights, oracle_mm, sample_cols, to_dev_bf16)
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

FAMILIES = ["auto", "simt", "tc", "vanilla"]


def _run(M, N, K, kernel="auto", seed=0, xseed=1):
    hw = host_weights(seed, N, K)
    w = dev_weights(seed, N, K)
    xb = synth.make_x(xseed, M, K)
    y = ops.mm(to_dev_bf16(xb), w, kernel=kernel)
    torch.cuda.synchronize()
    return xb, hw, y


@pytest.mark.parametrize("kernel", FAMILIES)
def test_tiny_matvec_full(kernel):
    N, K = TINY
    xb, hw, y = _run(1, N, K, kernel, xseed=0)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"tiny {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "vanilla"])
@pytest.mark.parametrize("N,K", [(1, 64), (7, 128), (9, 192), (31, 1088), (33, 2560), (129, 640), (1000, 3072)])
@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_ragged_shapes(kernel, N, K, M):
    xb, hw, y = _run(M, N, K, kernel, seed=N + K, xseed=M)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"{kernel} M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(1, 512), (7, 1024), (31, 1536), (33, 2560), (95, 1536), (1000, 3072), (4099, 4096)])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 13])
def test_tc_ragged_shapes(N, K, M):
    xb, hw, y = _run(M, N, K, "tc", seed=N + K + 1, xseed=M + 40)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"tc M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(1, 512), (7, 1024), (31, 1536), (33, 2560), (95, 1536), (1000, 3072), (4099, 4096)])
@pytest.mark.parametrize("M", [1, 5, 8])
def test_tc_persistent_grid_ragged_shapes(N, K, M):
    """The persistent launch shape without a workspace (units dealt inside each
    CTA; a split K as whole-K units folding the slice sums), forced on shapes
    the dispatcher would give to the tile kernel."""
    xb, hw, y = _run(M, N, K, "tc_stream", seed=N + K + 1, xseed=M + 40)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"tc_stream M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(1, 512), (31, 1536), (1000, 3072), (2560, 10240), (1536, 12288)])
@pytest.mark.parametrize("M", [1, 3])
def test_tc_tile_kernel_ragged_shapes(N, K, M):
    """The tile launch shape, forced on shapes the dispatcher may give to the
    persistent grid (more CTAs than fit at once run in waves)."""
    xb, hw, y = _run(M, N, K, "tc_tile", seed=N + K + 2, xseed=M + 50)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"tc_tile M={M} N={N} K={K}")


def test_tc_takes_k_not_multiple_of_512_up_to_its_slot_limit():
    """K % 512 != 0 runs on the tensor cores padded to whole stages while the
    per-unit parameter rows fit in shared memory; past that, only on request
    of another family."""
    xb, hw, y = _run(1, 64, 768, "tc")
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, "tc 64x768")
    with pytest.raises(ValueError):
        _run(1, 64, 6016, "tc")


def _special_case(N, K, codes, scale, bias, M=4):
    rng = np.random.default_rng(N * K)
    xb = synth.make_x(7, M, K)
    Wq = np.full((N, K // 8), codes, dtype=np.uint32)
    s = np.full((N, K // 64), scale, dtype=np.uint16)
    b = np.full((N, K // 64), bias, dtype=np.uint16)
    s[::2] ^= 0x8000  # negative scales on even rows
    host = synth.HostW4(Wq, s, b, N, K)
    yr, ad = oracle.mm(xb, Wq, s, b, M, N, K)
    return xb, host, yr, ad


@pytest.mark.parametrize("kernel", ["simt", "tc", "vanilla"])
@pytest.mark.parametrize("codes", [0x00000000, 0xFFFFFFFF, 0x87654321])
@pytest.mark.parametrize("K", [1536, 2304, 576])
def test_special_codes_and_signed_scales(kernel, codes, K):
    N = 77
    xb, host, yr, ad = _special_case(N, K, codes, 0x3C0E, 0xBDB4)  # s ~ 0.0087, b ~ -0.088
    y = ops.mm(to_dev_bf16(xb), ops.W4Matrix.from_host(host), kernel=kernel)
    assert_parity(y, yr, ad, f"codes {codes:#x}")


def test_empty_batch_writes_nothing():
    N, K = 64, 128
    w = dev_weights(0, N, K)
    y = torch.full((0, N), 3.0, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    out = ops.mm(x, w, out=y)
    assert out.shape == (0, N)


@pytest.mark.parametrize("name", sorted(DECODE_SET))
def test_decode_set_full(name):
    N, K = DECODE_SET[name]
    xb, hw, y = _run(1, N, K, seed=100 + sorted(DECODE_SET).index(name))
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"decode {name}")


@pytest.mark.parametrize("N,K", VERIFY_SHAPES)
@pytest.mark.parametrize("M", [1, 3, 5, 7])
def test_verify_shapes(N, K, M):
    xb, hw, y = _run(M, N, K, seed=3, xseed=11)
    cols = sample_cols(N, 2048, seed=M)
    yr, ad = oracle_mm(xb, hw, cols)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"verify {N}x{K} M={M}")


@pytest.mark.parametrize("N,K", LM_HEADS)
@pytest.mark.parametrize("M", [1, 3])
def test_lm_head_sampled(N, K, M):
    xb, hw, y = _run(M, N, K, seed=4, xseed=12)
    cols = sample_cols(N, 4096, seed=M)
    yr, ad = oracle_mm(xb, hw, cols)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"lm head {N}x{K} M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_dense_16k_sampled(M):
    N, K = DENSE
    xb, hw, y = _run(M, N, K, seed=5, xseed=13)
    cols = sample_cols(N, 1024, seed=M)
    yr, ad = oracle_mm(xb, hw, cols)
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"dense 16k M={M}")


def test_large_activation_magnitudes():
    N, K = 96, 2048
    hw = host_weights(9, N, K)
    rng = np.random.default_rng(3)
    xf = (rng.standard_normal((2, K)) * 1e15).astype(np.float32)
    xb = oracle.bf16_from_f32(xf)
    y = ops.mm(to_dev_bf16(xb), dev_weights(9, N, K))
    yr, ad = oracle.mm(xb, hw.Wq, hw.scales, hw.biases, 2, N, K)
    assert_parity(y, yr, ad, "x ~ 1e15")


def test_workspace_reuse_across_shapes():
    """Shapes of different sizes, split-K ones among them, share one stream's
    workspace (the binding's default); each call must find its counters at
    zero whatever ran before."""
    for (M, N, K) in [(2, 1024, 2560), (1, 12288, 8192), (3, 2560, 10240), (1, 98304, 1536), (5, 12288, 8192),
                      (4, 96, 1024), (1, 12288, 8192)]:
        xb, hw, y = _run(M, N, K, "auto", seed=N % 7, xseed=M)
        cols = sample_cols(N, 1024, seed=N)
        yr, ad = oracle_mm(xb, hw, cols)
        assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"reuse M={M} N={N} K={K}")
    assert ops.device_status() == 0
