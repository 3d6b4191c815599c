"""Lossless-verify invariance: row m of an M-row call equals the M = 1 call on
x[m], bit for bit ("Gemma 4 E4B & E2B -- single-launch Metal megakernels"
model card, "Measured performance": batch verify vs sequential, max abs diff
0.0).  Also routed rows vs the plain call on the chosen expert."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import (DECODE_SET, DENSE, EXPERTS, LM_HEADS, VERIFY_SHAPES, assert_parity, bf16_bits, dev_weights,
                       to_dev_bf16)
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _rows_equal_single(N, K, Ms, kernel="auto", seed=0):
    w = dev_weights(seed, N, K)
    Mmax = max(Ms)
    x = to_dev_bf16(synth.make_x(21, Mmax, K))
    singles = [bf16_bits(ops.mm(x[m:m + 1], w, kernel=kernel)) for m in range(Mmax)]
    for M in Ms:
        batch = bf16_bits(ops.mm(x[:M], w, kernel=kernel))
        for m in range(M):
            assert np.array_equal(batch[m], singles[m][0]), f"{N}x{K} {kernel}: row {m} of M={M} differs"


@pytest.mark.parametrize("N,K", VERIFY_SHAPES + [DECODE_SET["k"], DECODE_SET["o"], (33, 2560), (1, 64)])
def test_verify_rows_bitwise(N, K):
    _rows_equal_single(N, K, [2, 3, 4, 5, 6, 7, 8, 9, 16])


@pytest.mark.parametrize("kernel", ["simt", "tc", "vanilla"])
def test_every_family_is_batch_invariant(kernel):
    _rows_equal_single(1000, 3072, [3, 8, 11], kernel=kernel, seed=2)


@pytest.mark.parametrize("N,K", [(1, 512), (33, 2560), (1000, 3072), (4099, 4096), (12288, 1536), (6144, 2048)]
                         + sorted(set(DECODE_SET.values())))
def test_tc_launch_shapes_agree_bitwise(N, K):
    """The persistent grid and the tile kernel implement the same canonical
    slice order, so the dispatcher may pick either for any M."""
    w = dev_weights(6, N, K)
    x = to_dev_bf16(synth.make_x(24, 8, K))
    for M in (1, 3, 8):
        a = bf16_bits(ops.mm(x[:M], w, kernel="tc_stream"))
        try:
            b = bf16_bits(ops.mm(x[:M], w, kernel="tc_tile"))
        except ops.W4A16ValueError:
            assert M > 1, "the tile kernel holds every decode shape at M = 1"
            continue
        assert np.array_equal(a, b), f"{N}x{K} M={M}: tile and persistent launches differ"
        assert np.array_equal(a, bf16_bits(ops.mm(x[:M], w))), f"{N}x{K} M={M}: dispatcher differs"


def test_lm_head_rows_bitwise():
    N, K = LM_HEADS[0]
    _rows_equal_single(N, K, [3], seed=4)


def test_dense_rows_bitwise():
    N, K = DENSE
    _rows_equal_single(N, K, [2, 4, 8], seed=5)


def test_row_order_and_neighbours_do_not_matter():
    N, K = 2560, 10240
    w = dev_weights(3, N, K)
    x = to_dev_bf16(synth.make_x(22, 8, K))
    a = bf16_bits(ops.mm(x, w))
    perm = torch.tensor([5, 2, 7, 0, 1, 6, 3, 4], device="cuda")
    b = bf16_bits(ops.mm(x[perm].contiguous(), w))
    assert np.array_equal(a[perm.cpu().numpy()], b)


def test_n_sharding_concatenates_bitwise():
    """Splitting the output rows into independent launches (the multi-GPU
    sharding, run here on one GPU) reproduces the unsharded call exactly
    whenever a shard gets the same reduction plan (ksplit, slice_k) as the
    full matrix; every shard stays within the oracle tolerance regardless."""
    E_unused, N, K = EXPERTS
    hw = synth.make_weights(8, N, K)
    w = ops.W4Matrix.from_host(hw)
    xb = synth.make_x(23, 3, K)
    x = to_dev_bf16(xb)
    full = bf16_bits(ops.mm(x, w))
    full_plan = ops.get_plan(N, K)
    same_plan = 0
    for lo, hi in [(0, 1536), (1536, 4096), (4096, N), (0, 3072), (3072, N)]:
        shard = synth.HostW4(hw.Wq[lo:hi].copy(), hw.scales[lo:hi].copy(), hw.biases[lo:hi].copy(), hi - lo, K)
        part = bf16_bits(ops.mm(x, ops.W4Matrix.from_host(shard)))
        pl = ops.get_plan(hi - lo, K)
        if (pl["ksplit"], pl["slice_k"]) == (full_plan["ksplit"], full_plan["slice_k"]):
            same_plan += 1
            assert np.array_equal(part, full[:, lo:hi]), f"shard {lo}:{hi}"
        else:
            yr, ad = oracle.mm(xb, shard.Wq, shard.scales, shard.biases, 3, hi - lo, K)
            assert_parity(torch.from_numpy(part.view(np.int16)).view(torch.bfloat16), yr, ad, f"shard {lo}:{hi}")
    assert same_plan >= 1


def test_mm_id_rows_equal_mm_on_selected_expert():
    E, N, K = EXPERTS
    hw = synth.make_weights(30, N, K, E)
    w = ops.W4Matrix.from_host(hw)
    T = 13
    ids_np = synth.make_ids(30, T, E)
    ids = torch.from_numpy(ids_np).cuda()
    x = to_dev_bf16(synth.make_x(31, T, K))
    y = bf16_bits(ops.mm_id(x, w, ids))
    for t in range(T):
        e = int(ids_np[t])
        we = ops.W4Matrix(w.Wq[e].contiguous(), w.scales[e].contiguous(), w.biases[e].contiguous(), N, K)
        ref = bf16_bits(ops.mm(x[t:t + 1], we))
        assert np.array_equal(y[t], ref[0]), f"token {t} (expert {e})"


@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240), (300, 1024)])
def test_many_rows_one_launch(N, K):
    """More than eight rows in one tile-kernel launch (the rows stream through
    in chunks of eight over resident weights): every row bitwise equal to its
    M = 1 call and within tolerance of the oracle; the persistent launch shape
    (a launch per chunk) gives the same bits."""
    hw_seed = 4
    w = dev_weights(hw_seed, N, K)
    M = 37
    xb = synth.make_x(33, M, K)
    x = to_dev_bf16(xb)
    y = bf16_bits(ops.mm(x, w))
    assert np.array_equal(y, bf16_bits(ops.mm(x, w, kernel="tc_stream")))
    for m in (0, 7, 8, 9, 31, 32, 36):
        assert np.array_equal(y[m], bf16_bits(ops.mm(x[m:m + 1], w))[0]), f"row {m}"
    from gpu_cases import host_weights, oracle_mm, sample_cols
    cols = sample_cols(N, 256)
    yr, ad = oracle_mm(xb, host_weights(hw_seed, N, K), cols=cols)
    yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
    assert_parity(yt[:, torch.from_numpy(cols).cuda()], yr, ad, f"{N}x{K} M={M}")
