"""Programmatic dependent launch: a kernel may start (and fetch its weights)
while the previous kernel on the stream still runs, but reads activations
and ids, and writes outputs and the workspace, only after that kernel is
done.  Chains where each call consumes the previous call's output must give
the same bits with and without the overlap, eagerly and in a CUDA graph."""
import os

import numpy as np
import pytest
import torch

from gpu_cases import bf16_bits, dev_weights, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _set_pdl(mode):
    if mode is None:
        os.environ.pop("W4A16_PDL", None)
    else:
        os.environ["W4A16_PDL"] = str(mode)
    ops.lib().w4a16_debug_reload_env()


@pytest.fixture
def restore_pdl():
    yield
    _set_pdl(None)


# Each stage consumes the previous output: tile kernel, persistent split-K,
# tile kernel with M > 1, persistent single-slice, then routed experts.
CHAIN = [(10240, 2560), (2560, 10240), (2048, 2560), (6144, 2048)]


def _chain(x, ws, wexp, ids, bufs, fill):
    h = x
    for w, out in zip(ws, bufs[:-1]):
        out.fill_(fill)
        ops.mm(h, w, out=out)
        h = out
    ybuf = bufs[-1]
    ybuf.fill_(fill)
    ids.copy_(torch.remainder(torch.arange(ids.numel(), device="cuda", dtype=torch.int32) * 5 + 3, 8))
    ops.mm_id(h, wexp, ids, out=ybuf)
    return [bf16_bits(b) for b in bufs]


def _setup(M):
    ws = [dev_weights(40 + i, N, K) for i, (N, K) in enumerate(CHAIN[:3])]
    wexp = ops.W4Matrix.from_host(synth.make_weights(44, 6144, 2048, 8))
    x = to_dev_bf16(synth.make_x(45, M, 2560))
    bufs = [torch.empty(M, w.N, dtype=torch.bfloat16, device="cuda") for w in ws]
    bufs.append(torch.empty(M, 6144, dtype=torch.bfloat16, device="cuda"))
    ids = torch.zeros(M, dtype=torch.int32, device="cuda")
    return x, ws, wexp, ids, bufs


@pytest.mark.parametrize("M", [1, 5])
def test_dependent_chain_matches_plain_launches(M, restore_pdl):
    x, ws, wexp, ids, bufs = _setup(M)
    _set_pdl(0)
    ref = _chain(x, ws, wexp, ids, bufs, float("nan"))
    for mode in (1, 2):
        _set_pdl(mode)
        for fill in (float("nan"), 0.0, -3.0):
            got = _chain(x, ws, wexp, ids, bufs, fill)
            for i, (a, b) in enumerate(zip(ref, got)):
                assert np.array_equal(a, b), f"PDL mode {mode}, fill {fill}: stage {i} differs"


def test_dependent_chain_in_cuda_graph(restore_pdl):
    M = 3
    x, ws, wexp, ids, bufs = _setup(M)
    _set_pdl(0)
    ref = _chain(x, ws, wexp, ids, bufs, float("nan"))
    _set_pdl(2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain(x, ws, wexp, ids, bufs, 1.0)  # first calls (workspace, attributes) outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            h = x
            for w, out in zip(ws, bufs[:-1]):
                ops.mm(h, w, out=out)
                h = out
            ops.mm_id(h, wexp, ids, out=bufs[-1])
    for fill in (float("nan"), 7.0):
        for b in bufs:
            b.fill_(fill)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(ref, [bf16_bits(b) for b in bufs])):
            assert np.array_equal(a, b), f"graph replay, fill {fill}: stage {i} differs"
