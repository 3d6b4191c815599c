"""A bounded device wait that runs out, on the GPU, without faulting it.

The debug switch W4A16_FAULT=wait makes one stage of one warp of the
persistent kernel expect 16 bytes more than its copies deliver.  Every copy
still lands, so nothing is in flight when that warp's wait gives up: the
kernel raises W4A16_DEVICE_TIMEOUT, waits (bounded) for its copies, exits,
and the CUDA context keeps working.  No trap, no bad address, no endless
loop is involved.
"""
import os
import time

import pytest
import torch

from gpu_cases import assert_parity, dev_weights, host_weights, oracle_mm, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 2


@pytest.fixture()
def wait_fault(monkeypatch):
    L = ops.lib()
    monkeypatch.setenv("W4A16_FAULT", "wait")
    L.w4a16_debug_reload_env()
    yield
    monkeypatch.delenv("W4A16_FAULT", raising=False)
    L.w4a16_debug_reload_env()


def _call(N, K, M, seed):
    w = dev_weights(seed, N, K)
    xb = synth.make_x(seed, M, K)
    return xb, ops.mm(to_dev_bf16(xb), w, kernel="tc_stream", workspace=None)


def test_wait_runs_out_and_the_context_survives(wait_fault):
    N, K, M = 256, 1024, 2
    assert ops.device_status() == 0
    t0 = time.perf_counter()
    _call(N, K, M, 5)
    flags = ops.device_status()  # synchronises: the kernel has ended
    elapsed = time.perf_counter() - t0
    assert flags & DEVICE_TIMEOUT, f"flags {flags:#x}: the planted wait did not run out"
    assert elapsed < 60, f"the bounded waits took {elapsed:.1f} s"
    # the same process, the switch off: normal calls give oracle results
    os.environ.pop("W4A16_FAULT", None)
    ops.lib().w4a16_debug_reload_env()
    xb, y = _call(N, K, M, 5)
    torch.cuda.synchronize()
    yr, ad = oracle_mm(xb, host_weights(5, N, K))
    assert_parity(y, yr, ad, "after a wait timeout")
    assert ops.device_status() == 0
    # and a large call on the other kernels too
    xb2, y2 = _call(16384, 16384, 1, 6)
    torch.cuda.synchronize()
    assert torch.isfinite(y2.float()).all()
    assert ops.device_status() == 0
