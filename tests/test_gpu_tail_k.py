"""K % 512 != 0 on the tensor-core kernels.

The tensor-core kernels stream 512-code stages; a K that is not a multiple of
512 (K % 64 == 0, e.g. hidden 2304 of the Gemma-2-sized LM head 256000x2304)
runs on the persistent kernel as K padded to whole stages, in whole-K work
units whose scale and bias rows come by bulk copy (rows K / 32 bytes apart fit
no tensor map).  The padding groups read zero codes (the tensor copies'
out-of-bounds fill), zero activations and parameters masked to zero, so they
add +0 to every slice partial.  Checked here: parity with the oracle element
by element (the oracle sums over the real K only), M rows against M = 1 bit
for bit, routed rows against w4a16_mm on their expert, that no activation or
parameter past a row is used (an inf at the start of the next row leaves a row
finite and unchanged), and the K range: up to 5952 on the tensor cores, the
CUDA-core family above.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_parity, bf16_bits, dev_weights, host_weights, oracle_mm, sample_cols, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

# ragged N; K one group, a few groups, just past a stage, and mid-stage tails
TAIL = [(1, 64), (7, 128), (9, 192), (31, 1088), (129, 640), (33, 2304), (1000, 2304), (95, 1600), (4099, 4160)]
LM_HEAD_TAIL = (256000, 2304)


@pytest.mark.parametrize("N,K", TAIL)
@pytest.mark.parametrize("M", [1, 2, 5, 8, 13])
def test_tail_k_parity(N, K, M):
    hw = host_weights(N + K + 3, N, K)
    w = dev_weights(N + K + 3, N, K)
    xb = synth.make_x(M + 50, M, K)
    assert ops.get_plan(N, K)["kernel"] == "tc"
    y = ops.mm(to_dev_bf16(xb), w)
    yr, ad = oracle_mm(xb, hw)
    assert_parity(y, yr, ad, f"tail K tc M={M} N={N} K={K}")
    assert ops.device_status() == 0


@pytest.mark.parametrize("N,K", TAIL + [(300, 5952), (2048, 2304)])
def test_tail_k_launch_shapes(N, K):
    """The dispatcher, the persistent kernel (whole-K units without a
    workspace, split with one at M = 1) and the tile kernel give the same bits;
    the prefill kernel refuses."""
    w = dev_weights(N + K + 3, N, K)
    x = to_dev_bf16(synth.make_x(77, 8, K))
    for M in (1, 3, 8):
        a = bf16_bits(ops.mm(x[:M], w, kernel="tc_stream"))
        assert np.array_equal(a, bf16_bits(ops.mm(x[:M], w))), f"{N}x{K} M={M}: dispatcher differs"
        assert np.array_equal(a, bf16_bits(ops.mm(x[:M], w, workspace=None))), f"{N}x{K} M={M}: no workspace"
        ws = ops.workspace()
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        args = (x[:M].data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), y.data_ptr(), M, N, K)
        assert ops.lib().w4a16_mm_ws(*args, *ops._ws_args(ws), None) == ops.OK
        assert np.array_equal(a, bf16_bits(y)), f"{N}x{K} M={M}: with a workspace"
        try:
            b = bf16_bits(ops.mm(x[:M], w, kernel="tc_tile"))
        except ops.W4A16ValueError:
            assert M > 1, "the tile kernel holds these shapes at M = 1"
            continue
        assert np.array_equal(a, b), f"{N}x{K} M={M}: tile and persistent launches differ"
    with pytest.raises(ValueError):
        ops.mm(x[:1], w, kernel="tc_prefill")


@pytest.mark.parametrize("N,K", [(9216, 2304), (3000, 5952)])
def test_tail_k_rows_bitwise(N, K):
    w = dev_weights(8, N, K)
    x = to_dev_bf16(synth.make_x(23, 16, K))
    singles = [bf16_bits(ops.mm(x[m:m + 1], w)) for m in range(16)]
    for M in (2, 3, 5, 8, 9, 16):
        batch = bf16_bits(ops.mm(x[:M], w))
        for m in range(M):
            assert np.array_equal(batch[m], singles[m][0]), f"{N}x{K}: row {m} of M={M} differs"


def test_tail_k_prefill_rows():
    """More than 32 rows (the prefill kernel's range when K % 512 == 0; here the
    persistent kernel, eight rows a launch): parity, and rows equal to the
    M = 1 calls."""
    N, K = 1000, 2304
    hw, w = host_weights(9, N, K), dev_weights(9, N, K)
    for M in (40, 130):
        xb = synth.make_x(M, M, K)
        x = to_dev_bf16(xb)
        y = ops.mm(x, w)
        yr, ad = oracle_mm(xb, hw)
        assert_parity(y, yr, ad, f"tail K prefill M={M}")
        rows = [0, 1, 31, 32, M - 1]
        ones = torch.stack([ops.mm(x[m:m + 1], w)[0] for m in rows])
        assert torch.equal(y[rows].view(torch.int16), ones.view(torch.int16)), f"M={M}: rows differ from M = 1"
    assert ops.device_status() == 0


def test_tail_k_lm_head():
    """The 256000x2304 LM head: sampled columns against the oracle at M = 3,
    rows of M = 3 equal to M = 1; w4a16_mm_argmax refuses K % 512 != 0."""
    N, K = LM_HEAD_TAIL
    hw, w = host_weights(12, N, K), dev_weights(12, N, K)
    xb = synth.make_x(12, 3, K)
    x = to_dev_bf16(xb)
    y3 = ops.mm(x, w)
    cols = sample_cols(N, 1024, seed=12)
    yr, ad = oracle_mm(xb, hw, cols)
    assert_parity(y3[:, torch.from_numpy(cols).cuda()], yr, ad, "tail K LM head M=3")
    for m in range(3):
        assert torch.equal(ops.mm(x[m:m + 1], w)[0].view(torch.int16), y3[m].view(torch.int16)), f"row {m}"
    with pytest.raises(ValueError):
        ops.mm_argmax(x, w)
    assert ops.device_status() == 0


@pytest.mark.parametrize("N,K", [(500, 2304), (7, 192), LM_HEAD_TAIL])
@pytest.mark.parametrize("kernel", ["tc_stream", "tc_tile", "tc_prefill", None])
def test_tail_k_reads_no_activation_past_k(N, K, kernel):
    """Row 1 starts with +inf: a kernel that took its padding activations from
    the next row would turn row 0 into NaN (0 * inf).  Rows 0 and 2 must stay
    finite and equal their M = 1 calls."""
    w = dev_weights(N + 1, N, K)
    xb = synth.make_x(31, 3, K).copy()
    xb[1, :64] = 0x7F80  # bf16 +inf
    x = to_dev_bf16(xb)
    try:
        y = ops.mm(x, w, kernel=kernel)
    except ops.W4A16ValueError:
        assert kernel == "tc_prefill" or (kernel == "tc_tile" and N * K > 10**8)
        return
    for m in (0, 2):
        assert torch.isfinite(y[m].float()).all(), f"row {m} not finite"
        assert torch.equal(y[m].view(torch.int16), ops.mm(x[m:m + 1], w)[0].view(torch.int16))


@pytest.mark.parametrize("E,N,K", [(1, 300, 2304), (1, 77, 576), (3, 201, 576), (2, 33, 1152)])
def test_tail_k_reads_no_parameter_past_a_row(E, N, K):
    """The parameter rows lie K / 32 bytes apart, so the bytes after a row's
    last group are the next row's first scales and biases; in the padded last
    stage they must read as zero.  With +inf there (the first scale and bias of
    every odd row), the even rows stay finite and within the oracle's bound
    (0 * inf would give NaN)."""
    hw = synth.make_weights(K + N, N, K, E)
    s = hw.scales.copy().reshape(E * N, K // 64)
    b = hw.biases.copy().reshape(E * N, K // 64)
    s[1::2, 0] = 0x7F80
    b[1::2, 0] = 0x7F80
    hw2 = synth.HostW4(hw.Wq, s.reshape(hw.scales.shape), b.reshape(hw.biases.shape), N, K, E)
    w = ops.W4Matrix.from_host(hw2)
    T = 6
    xb = synth.make_x(K, T, K)
    x = to_dev_bf16(xb)
    if E == 1:
        y = ops.mm(x, w)
        yr, ad = oracle.mm(xb, hw2.Wq, hw2.scales, hw2.biases, T, N, K, threads=oracle.host_threads())
    else:
        ids_np = np.arange(T, dtype=np.int32) % E
        y = ops.mm_id(x, w, torch.from_numpy(ids_np).cuda())
        yr, ad = oracle.mm_id(xb, hw2.Wq, hw2.scales, hw2.biases, ids_np, T, N, K, E)
    # rows whose stacked index is even: every row of an expert when N is even,
    # alternate rows otherwise
    ids = np.zeros(T, dtype=np.int64) if E == 1 else np.arange(T) % E
    for t in range(T):
        keep = ((ids[t] * N + np.arange(N)) % 2) == 0
        assert_parity(y[t][torch.from_numpy(np.nonzero(keep)[0]).cuda()], yr[t][keep], ad[t][keep], f"row {t}")


@pytest.mark.parametrize("kernel", ["auto", "tc_stream"])
@pytest.mark.parametrize("E,N,K,T", [(4, 640, 2304, 8), (3, 201, 576, 37), (8, 3000, 2304, 8), (5, 77, 1152, 70)])
def test_tail_k_routed(kernel, E, N, K, T):
    """w4a16_mm_id on K % 512 != 0 (experts whose parameter rows start off
    16-byte boundaries, more than 32 tokens): the oracle, and every token's
    row equal to w4a16_mm on its expert bit for bit."""
    hw = synth.make_weights(E + N, N, K, E)
    w = ops.W4Matrix.from_host(hw)
    ids_np = synth.make_ids(E, T, E)
    xb = synth.make_x(E, T, K)
    x = to_dev_bf16(xb)
    y = ops.mm_id(x, w, torch.from_numpy(ids_np).cuda(), kernel=kernel)
    cols = sample_cols(N, 512, seed=E)
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E, cols=cols,
                          threads=oracle.host_threads())
    assert_parity(y[:, torch.from_numpy(cols).cuda()], yr, ad, f"tail K mm_id {kernel}")
    for e in sorted(set(ids_np.tolist())):
        # a copy: an expert's tables inside the stack need not start on the
        # 8-byte boundary w4a16_mm asks of its own arguments
        we = ops.W4Matrix(w.Wq[e].clone(), w.scales[e].clone(), w.biases[e].clone(), N, K)
        toks = np.nonzero(ids_np == e)[0]
        ref = ops.mm(x[torch.from_numpy(toks).cuda()], we)
        assert torch.equal(y[torch.from_numpy(toks).cuda()].view(torch.int16), ref.view(torch.int16)), f"expert {e}"
    assert ops.device_status() == 0


def test_tail_k_routed_bad_ids():
    E, N, K, T = 4, 90, 1152, 9
    hw = synth.make_weights(3, N, K, E)
    w = ops.W4Matrix.from_host(hw)
    ids_np = np.array([1, -1, 3, 7, 1, 0, 2, 99, 3], dtype=np.int32)
    xb = synth.make_x(3, T, K)
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.mm_id(to_dev_bf16(xb), w, torch.from_numpy(ids_np).cuda(), out=y)
    assert ops.device_status() & ops.DEVICE_BAD_ID
    yr, ad = oracle.mm_id(xb, hw.Wq, hw.scales, hw.biases, ids_np, T, N, K, E)
    assert_parity(y, yr, ad, "tail K bad ids")
    for t in (1, 3, 7):
        assert np.all(bf16_bits(y)[t] == 0)


@pytest.mark.parametrize("N,K,kernel", [(300, 5952, "tc"), (300, 6016, "simt"), (2048, 6912, "simt")])
def test_tail_k_range(N, K, kernel):
    """The largest K % 512 != 0 the persistent kernel's per-unit parameter
    slots hold (next to a two-stage ring with eight activation rows) is 5952;
    larger ones run on the CUDA-core family.  Both pass parity."""
    assert ops.get_plan(N, K)["kernel"] == kernel
    hw, w = host_weights(N + 5, N, K), dev_weights(N + 5, N, K)
    for M in (1, 8):
        xb = synth.make_x(M, M, K)
        y = ops.mm(to_dev_bf16(xb), w)
        yr, ad = oracle_mm(xb, hw)
        assert_parity(y, yr, ad, f"{kernel} M={M} N={N} K={K}")
