"""The library allocates nothing: w4a16_mm runs without a workspace, and
w4a16_mm_ws with the caller's one, with the same bits.

Without a workspace the persistent grid deals its units inside each CTA and
a K split across SMs becomes either the tile kernel's clusters (slice sums in
distributed shared memory) or whole-K units that fold the slice sums in
registers; with one, a grid-wide unit counter and fp32 partials in the
workspace.  Every variant adds the same canonical slice sums in the same
order, so the outputs must agree bit for bit, and with the oracle within the
parity tolerance.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_cases import DENSE, LM_HEADS, assert_parity, dev_weights, host_weights, oracle_mm, sample_cols, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (N, K): persistent-grid shapes with K split across SMs (ksplit > 1), one
# without a split, and the LM head.
SPLIT_SHAPES = [DENSE, (16384, 8192)]
NOSPLIT_SHAPE = (98304, 1536)


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("N,K", SPLIT_SHAPES + [NOSPLIT_SHAPE, LM_HEADS[1]])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_with_and_without_workspace_agree_bitwise(N, K, M):
    plan = ops.get_plan(N, K)
    assert plan["workspace_bytes"] > 0, "a persistent-grid shape"
    w = dev_weights(31, N, K)
    xb = synth.make_x(32 + M, M, K)
    x = to_dev_bf16(xb)
    y_ws = ops.mm(x, w)                                 # w4a16_mm_ws, this stream's workspace
    y_none = ops.mm(x, w, workspace=None)               # w4a16_mm
    y_stream = ops.mm(x, w, kernel="tc_stream")          # the persistent grid without a workspace
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_ws), _bits(y_none)), f"w4a16_mm vs w4a16_mm_ws, M={M} N={N} K={K}"
    assert torch.equal(_bits(y_ws), _bits(y_stream)), f"persistent grid without a workspace, M={M} N={N} K={K}"
    if M == 3:
        cols = sample_cols(N, 512, seed=N + K)
        yr, ad = oracle_mm(xb, host_weights(31, N, K), cols)
        assert_parity(y_none[:, torch.from_numpy(cols).cuda()], yr, ad, f"no workspace M={M} N={N} K={K}")
    assert ops.device_status() == 0


def test_split_shapes_use_the_split():
    for N, K in SPLIT_SHAPES:
        assert ops.get_plan(N, K)["ksplit"] > 1
    assert ops.get_plan(*NOSPLIT_SHAPE)["ksplit"] == 1


def test_no_device_memory_taken_by_calls():
    """After one warm-up call (module loading), w4a16_mm calls on a stream
    the library has not seen change nothing in the device's free memory.
    The stream is made before the first reading: torch's first stream
    creation sets up its stream pool, which takes device memory of its own."""
    shapes = SPLIT_SHAPES + [NOSPLIT_SHAPE]
    ws = [dev_weights(31, N, K) for N, K in shapes]
    xs = [to_dev_bf16(synth.make_x(40, 2, K)) for _, K in shapes]
    ys = [torch.empty(2, N, dtype=torch.bfloat16, device="cuda") for N, _ in shapes]
    for x, w, y in zip(xs, ws, ys):
        ops.mm(x, w, out=y, workspace=None)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(s):
        for _ in range(3):
            for x, w, y in zip(xs, ws, ys):
                ops.mm(x, w, out=y, workspace=None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


_FIRST_CALL_IN_CAPTURE = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from skinny_gemm_gb300 import ops, synth

torch.cuda.set_device(0)
out = []
for (N, K) in [(16384, 16384), (98304, 1536), (2048, 2560)]:
    w = ops.W4Matrix.from_host(synth.make_weights(5, N, K))
    x = torch.from_numpy(synth.make_x(6, 2, K).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.full((2, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):   # the library's first call on this stream (and, for the first shape, ever)
        ops.mm(x, w, out=y, workspace=None)
    g.replay()
    torch.cuda.synchronize()
    ref = ops.mm(x, w, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (N, K)
    out.append(f"{N}x{K}")
print("captured first calls:", " ".join(out))
"""


def test_first_call_is_captured_into_a_cuda_graph():
    """A fresh process whose first library call is made while its stream is
    captured: nothing to allocate, so the capture succeeds and the replay
    gives the eager call's bits."""
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "captured first calls" in r.stdout


def test_caller_workspace_is_left_zeroed():
    """A caller-owned workspace: zeroed once, shared by calls of several
    shapes on one stream, and zero again after they complete."""
    nb = ops.workspace_bytes(*DENSE)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    shapes = SPLIT_SHAPES + [NOSPLIT_SHAPE, LM_HEADS[1]]
    for i, (N, K) in enumerate(shapes * 2):
        w = dev_weights(31, N, K)
        x = to_dev_bf16(synth.make_x(50 + i, 1 + i % 5, K))
        a = ops.mm(x, w, workspace=ws)
        b = ops.mm(x, w, workspace=None)
        torch.cuda.synchronize()
        assert torch.equal(_bits(a), _bits(b)), (N, K)
    torch.cuda.synchronize()
    counters = ws[:32768].view(torch.int32)
    assert int(counters.abs().sum()) == 0
