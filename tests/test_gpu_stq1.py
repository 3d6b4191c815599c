"""STQ1_0 ternary matmul on the GPU against the CPU oracle.

Format and kernels of "Hy4-preview Metal kernels for llama.cpp" (sections
"Notes and gotchas" and the kernel table): matvec and small batches
(stq1_mm), routed experts (stq1_mm_id), the row gather (stq1_get_rows).
Inputs come from the seeded generator with the page's shapes (6144x2048
experts, the 16384x16384 matvec); expected values only from the oracle.
Bound: |y - y_ref| <= (2^-16 + (K/256 + 16) 2^-23) sum_k |x w| element by
element (oracle.stq1_tolerance); rows of a multi-row call must equal the
one-row call bit for bit, routed rows the plain call on their expert.
"""
import numpy as np
import pytest
import torch

import oracle
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def dev_x(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def check(y: torch.Tensor, yr: np.ndarray, ad: np.ndarray, K: int, what: str):
    got = y.double().cpu().numpy()
    err = np.abs(got - yr)
    tol = oracle.stq1_tolerance(ad, K)
    worst = int(np.argmax((err - tol).ravel()))
    assert np.all(err <= tol), (f"{what}: |y - y_ref| = {err.ravel()[worst]:.3e} > {tol.ravel()[worst]:.3e} "
                                f"at flat index {worst}")


@pytest.mark.parametrize("N,K,M", [(1, 256, 2), (7, 512, 1), (16, 256, 1), (20, 512, 1), (70, 512, 3),
                                   (300, 2048, 5), (1000, 4096, 8), (37, 1024, 11), (129, 768, 2), (6144, 2048, 1),
                                   (6144, 2048, 4)])
def test_parity_full(N, K, M):
    """Ragged row tiles (N % 16 != 0, down to one row), K = 1..16 blocks, K
    split over clusters of 1 to 8 CTAs, one to eight rows, and two passes
    (M = 11)."""
    blocks = synth.make_stq1(N + K, N, K)
    x = synth.make_x_f32(M, M, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    y = ops.stq1_mm(dev_x(x), w)
    yr, ad = oracle.stq1_mm(x, blocks, M, N, K, threads=oracle.host_threads())
    check(y, yr, ad, K, f"{N}x{K} M={M}")


@pytest.mark.parametrize("M", [1, 2, 3])
def test_parity_16384_sampled(M):
    """The page's 16384x16384 matvec (and two and three rows), sampled output
    columns in every 16-row tile position (four K slices of 16 blocks)."""
    N = K = 16384
    blocks = synth.make_stq1(16, N, K)
    x = synth.make_x_f32(160 + M, M, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    y = ops.stq1_mm(dev_x(x), w)
    cols = np.unique(np.concatenate([np.arange(0, N, 61), [N - 1, N - 16, 15, 16]]))
    yr, ad = oracle.stq1_mm(x, blocks, M, N, K, cols=cols, threads=oracle.host_threads())
    check(y[:, torch.from_numpy(cols).cuda()], yr, ad, K, f"16384^2 M={M}")


@pytest.mark.parametrize("N,K,M", [(6144, 2048, 8), (1000, 4096, 7), (16384, 16384, 5), (37, 1024, 11)])
def test_rows_equal_one_row_calls(N, K, M):
    blocks = synth.make_stq1(3, N, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    x = dev_x(synth.make_x_f32(30 + M, M, K))
    y = ops.stq1_mm(x, w)
    for m in range(M):
        y1 = ops.stq1_mm(x[m:m + 1].contiguous(), w)
        assert torch.equal(y[m:m + 1].view(torch.int32), y1.view(torch.int32)), f"row {m} of {M} differs from M = 1"


def test_closed_forms():
    """All-zero blocks give exact zeros; code 0 with no signs and d = 1 against
    x = 1 gives exactly 192 per block (lanes 1..3 of 64 groups), all signs set
    gives -192 per block."""
    N, K = 48, 1024
    zero = np.zeros((N, K // 256, 42), dtype=np.uint8)
    x = torch.ones(3, K, device="cuda")
    assert torch.count_nonzero(ops.stq1_mm(x, ops.STQ1Matrix.from_host(zero, N, K))) == 0
    one = zero.copy()
    one[:, :, 40], one[:, :, 41] = 0x00, 0x3C  # fp16 1.0
    assert torch.all(ops.stq1_mm(x, ops.STQ1Matrix.from_host(one, N, K)) == 192.0 * (K // 256))
    one[:, :, 32:40] = 0xFF
    assert torch.all(ops.stq1_mm(x, ops.STQ1Matrix.from_host(one, N, K)) == -192.0 * (K // 256))


def test_mm_id_page_workload():
    """Eight distinct 6144x2048 experts, eight tokens with uniform ids: against
    the oracle, and each row equal to stq1_mm on its expert bit for bit."""
    E, N, K, T = 8, 6144, 2048, 8
    blocks = synth.make_stq1(0, N, K, E)
    ids_np = synth.make_ids(0, T, E)
    x = synth.make_x_f32(0, T, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K, E)
    xd, ids = dev_x(x), torch.from_numpy(ids_np).cuda()
    y = ops.stq1_mm_id(xd, w, ids)
    yr, ad = oracle.stq1_mm_id(x, blocks, ids_np, T, N, K, E, threads=oracle.host_threads())
    check(y, yr, ad, K, "routed 8 x 6144x2048")
    per = ops.stq1_packed_bytes(N, K)
    for t in range(T):
        e = int(ids_np[t])
        we = ops.STQ1Matrix(w.packed[e * per:(e + 1) * per], N, K)
        assert torch.equal(y[t].view(torch.int32), ops.stq1_mm(xd[t:t + 1].contiguous(), we)[0].view(torch.int32))
    assert ops.device_status() == 0


@pytest.mark.parametrize("T,K", [(37, 1024), (20, 16384)])
def test_mm_id_many_tokens_one_expert(T, K):
    """More tokens on one expert than one pass holds (passes inside the
    kernel), the others spread, one bad id (zero row and the device flag)."""
    E, N = 4, 200
    blocks = synth.make_stq1(5, N, K, E)
    ids_np = np.full(T, 2, dtype=np.int32)
    ids_np[::5] = 1
    ids_np[3] = 7
    x = synth.make_x_f32(5, T, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K, E)
    y = ops.stq1_mm_id(dev_x(x), w, torch.from_numpy(ids_np).cuda())
    assert ops.device_status() == ops.DEVICE_BAD_ID
    yr, ad = oracle.stq1_mm_id(x, blocks, ids_np, T, N, K, E, threads=oracle.host_threads())
    check(y, yr, ad, K, f"routed T={T} K={K}")
    assert torch.count_nonzero(y[3]) == 0


def test_get_rows_exact():
    N, K = 300, 2560 // 256 * 256
    blocks = synth.make_stq1(8, N, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    ids_np = np.array([0, 299, 17, 16, 15, 150, -1, 300, 17], dtype=np.int32)
    rows = ops.stq1_get_rows(torch.from_numpy(ids_np).cuda(), w)
    assert ops.device_status() == ops.DEVICE_BAD_ID
    want = oracle.stq1_get_rows(blocks, ids_np, N, K)
    assert np.array_equal(rows.cpu().numpy(), want), "rows differ from the oracle's d * v"


def test_graph_capture_and_streams():
    N, K, M = 6144, 2048, 2
    w = ops.STQ1Matrix.from_host(synth.make_stq1(9, N, K), N, K)
    x = dev_x(synth.make_x_f32(9, M, K))
    want = ops.stq1_mm(x, w)
    out = torch.empty_like(want)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ops.stq1_mm(x, w, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.stq1_mm(x, w, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), want.view(torch.int32))


def test_mm_id_many_experts_grid_per_expert():
    """E > 1024 experts: one grid column per expert instead of the dealt
    units (two-tile matrices keep the weights at 1100 x 1344 bytes)."""
    E, N, K, T = 1100, 20, 256, 9
    blocks = synth.make_stq1(13, N, K, E)
    ids_np = np.array([1099, 0, 517, 1099, 3, 1024, 1023, 0, 77], dtype=np.int32)
    x = synth.make_x_f32(13, T, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K, E)
    y = ops.stq1_mm_id(dev_x(x), w, torch.from_numpy(ids_np).cuda())
    yr, ad = oracle.stq1_mm_id(x, blocks, ids_np, T, N, K, E, threads=oracle.host_threads())
    check(y, yr, ad, K, "routed, 1100 experts")
    assert ops.device_status() == 0


def test_largest_k():
    """K = 32768: eight slices of 16 blocks, three rows in one pass."""
    N, K, M = 40, 32768, 3
    assert ops.stq1_get_plan(N, K) == {"ksplit": 8, "blocks_per_slice": 16, "rows_per_pass": 8}
    blocks = synth.make_stq1(14, N, K)
    x = synth.make_x_f32(14, M, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    xd = dev_x(x)
    y = ops.stq1_mm(xd, w)
    yr, ad = oracle.stq1_mm(x, blocks, M, N, K, threads=oracle.host_threads())
    check(y, yr, ad, K, "K = 32768")
    assert torch.equal(y[1:2].view(torch.int32), ops.stq1_mm(xd[1:2].contiguous(), w).view(torch.int32))


CANARY32 = 0x7FA1C0DE  # a NaN pattern none of these kernels writes (finite inputs give finite outputs)
PAD = 2048


def _guarded(n: int):
    buf = torch.full((PAD + n + PAD,), CANARY32, dtype=torch.int32, device="cuda")
    return buf, buf[PAD:PAD + n].view(torch.float32)


def _check_guards(buf: torch.Tensor, n: int):
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:PAD] == CANARY32) and np.all(b[PAD + n:] == CANARY32), "write outside the output"
    assert not np.any(b[PAD:PAD + n] == CANARY32), "some outputs were not written"


@pytest.mark.parametrize("M,N,K", [(1, 37, 512), (3, 129, 2048), (11, 20, 1024), (2, 16, 16384)])
def test_output_guard_bands(M, N, K):
    """Outputs inside canary bands: ragged tiles, several passes, the largest split."""
    w = ops.STQ1Matrix.from_host(synth.make_stq1(70 + N, N, K), N, K)
    x = dev_x(synth.make_x_f32(70, M, K))
    buf, flat = _guarded(M * N)
    ops.stq1_mm(x, w, out=flat.view(M, N))
    _check_guards(buf, M * N)


def test_routed_and_row_gather_guard_bands():
    E, N, K, T = 3, 45, 512, 10
    w = ops.STQ1Matrix.from_host(synth.make_stq1(71, N, K, E), N, K, E)
    ids = torch.from_numpy(synth.make_ids(71, T, E)).cuda()
    x = dev_x(synth.make_x_f32(71, T, K))
    buf, flat = _guarded(T * N)
    ops.stq1_mm_id(x, w, ids, out=flat.view(T, N))
    _check_guards(buf, T * N)
    w0 = ops.STQ1Matrix(w.packed[:ops.stq1_packed_bytes(N, K)], N, K)
    rows = torch.tensor([44, 0, 17, 16, 3], dtype=torch.int32, device="cuda")
    buf, flat = _guarded(5 * K)
    ops.stq1_get_rows(rows, w0, out=flat.view(5, K))
    _check_guards(buf, 5 * K)
    assert ops.device_status() == 0


def test_extreme_activation_magnitudes():
    """Activations near the float32 range's ends: |x| up to 3e38 (one such
    value per group, so no table entry overflows) and around 2^-120 (float32
    additions keep subnormal values)."""
    N, K = 48, 512
    blocks = synth.make_stq1(31, N, K)
    w = ops.STQ1Matrix.from_host(blocks, N, K)
    rng = np.random.default_rng(5)
    x = np.zeros((3, K), dtype=np.float32)
    x[0, 7] = 3.0e38    # one value near the top of the range (a block sum of two such could overflow)
    x[0, 300] = -2.5e38  # another block
    x[1] = (rng.standard_normal(K) * 2.0 ** -120).astype(np.float32)
    x[2] = rng.standard_normal(K).astype(np.float32) * np.float32(1e30)
    y = ops.stq1_mm(dev_x(x), w)
    yr, ad = oracle.stq1_mm(x, blocks, 3, N, K)
    got = y.double().cpu().numpy()
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[2]))
    tol = oracle.stq1_tolerance(ad, K) + 2.0 ** -133 * K
    assert np.all(np.abs(got - yr) <= tol), float(np.max(np.abs(got - yr) - tol))
