"""w4a16_mm_noalloc: the entry point for callers that may not allocate device
memory (an engine that reserved all memory at start-up, a process under a
hard memory cap, a deployment that forbids allocation after initialisation).

It must give the same answer as w4a16_mm while keeping its split-K scratch in
a fixed array inside the library.  The array is shared by every call and
keeps the previous call's contents, so the test makes two calls in a row
(different shapes, so the second finds the first one's leftovers) and checks
each against w4a16_mm within the parity tolerance -- and, since both run the
same kernel, bit for bit.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc(x, w, y):
    L = ops.lib()
    M = x.numel() // w.K
    return L.w4a16_mm_noalloc(x.data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(),
                              y.data_ptr(), M, w.N, w.K, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_mm_on_two_calls_in_a_row():
    for (M, N, K, seed) in [(3, 10240, 2560, 71), (1, 2560, 10240, 72)]:
        # both shapes split K (so the scratch's counters and partials are used)
        assert ops.get_plan(N, K)["ksplit"] > 1
        hw = synth.make_weights(seed, N, K)
        w = ops.W4Matrix.from_host(hw)
        xb = synth.make_x(seed, M, K)
        x = _dev(xb)
        y_mm = ops.mm(x, w)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(x, w, y)
        assert rc == ops.OK, ops.lib().w4a16_last_error().decode()
        torch.cuda.synchronize()
        assert ops.device_status() == 0
        # tolerance of the parity tests, with the w4a16_mm output as the reference values
        _, absdot = oracle.mm(xb, hw.Wq, hw.scales, hw.biases, M, N, K, threads=oracle.host_threads())
        ref = y_mm.double().cpu().numpy()
        got = y.double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= oracle.tolerance(ref, absdot)), f"M={M} N={N} K={K}"
        assert torch.equal(y.view(torch.int16), y_mm.view(torch.int16)), "same kernel, same bits"


def test_noalloc_on_new_streams_takes_no_memory():
    """After one warm-up call (the library's module is loaded and the array's
    address looked up), calls on a brand-new stream leave the device's free
    memory unchanged, and a call captured on another new stream replays with
    w4a16_mm's bits."""
    M, N, K = 2, 2560, 10240
    hw = synth.make_weights(74, N, K)
    w = ops.W4Matrix.from_host(hw)
    x = _dev(synth.make_x(74, M, K))
    ref = ops.mm(x, w)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(x, w, y) == ops.OK
    # eager calls on a new stream: the device's free memory does not move
    # (the stream is made first: torch's first stream creation sets up its
    # stream pool, which takes device memory of its own)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(s):
        for _ in range(3):
            assert _noalloc(x, w, y) == ops.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    # captured on another new stream (an allocation would break the capture)
    s2 = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    y.fill_(float("nan"))
    torch.cuda.synchronize()
    rcs = []
    with torch.cuda.graph(g, stream=s2):
        rcs.append(_noalloc(x, w, y))
    assert rcs == [ops.OK], ops.lib().w4a16_last_error().decode()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("N,K", [(64, 192), (3000, 2304)])
def test_noalloc_takes_tail_k(N, K):
    """K % 512 != 0 (padded to whole stages) gives w4a16_mm's bits."""
    w = ops.W4Matrix.from_host(synth.make_weights(73, N, K))
    x = _dev(synth.make_x(73, 3, K))
    y = torch.empty(3, N, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(x, w, y) == ops.OK
    assert torch.equal(y.view(torch.int16), ops.mm(x, w, workspace=None).view(torch.int16))
