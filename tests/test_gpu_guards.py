"""Out-of-bounds writes and launch errors, detected without compute-sanitizer:
outputs live inside guard bands whose canary values must survive, and
rejected or fault-injected calls leave the output untouched."""
import numpy as np
import pytest
import torch

from gpu_cases import bf16_bits, dev_weights, to_dev_bf16
from skinny_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

CANARY = 0x7FA1  # a NaN pattern no kernel writes


@pytest.mark.parametrize("kernel", ["simt", "tc", "vanilla"])
@pytest.mark.parametrize("M,N,K", [(1, 7, 512), (5, 33, 2560), (9, 129, 1536), (3, 1000, 3072)])
def test_output_guard_bands(kernel, M, N, K):
    w = dev_weights(50 + N, N, K)
    x = to_dev_bf16(synth.make_x(50, M, K))
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 0, dtype=torch.int16, device="cuda")
    buf.fill_(CANARY)
    out = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    ops.mm(x, w, out=out, kernel=kernel)
    torch.cuda.synchronize()
    b = buf.cpu().numpy().view(np.uint16)
    assert np.all(b[:pad] == CANARY) and np.all(b[pad + M * N:] == CANARY), "write outside y"
    assert not np.any(b[pad:pad + M * N] == CANARY), "some outputs were not written"


def test_mm_id_guard_bands():
    E, N, K, T = 3, 45, 1024, 10
    hw = synth.make_weights(60, N, K, E)
    w = ops.W4Matrix.from_host(hw)
    ids = torch.from_numpy(synth.make_ids(60, T, E)).cuda()
    x = to_dev_bf16(synth.make_x(60, T, K))
    pad = 2048
    buf = torch.full((pad + T * N + pad,), CANARY, dtype=torch.int16, device="cuda")
    out = buf[pad:pad + T * N].view(torch.bfloat16).view(T, N)
    ops.mm_id(x, w, ids, out=out)
    b = buf.cpu().numpy().view(np.uint16)
    assert np.all(b[:pad] == CANARY) and np.all(b[pad + T * N:] == CANARY)
    assert not np.any(b[pad:pad + T * N] == CANARY)


def test_rejected_and_injected_calls_write_nothing(monkeypatch):
    N, K = 64, 128
    w = dev_weights(61, N, K)
    x = to_dev_bf16(synth.make_x(61, 2, K))
    y = torch.full((2, N), 5.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ops.mm(x[:, :64].contiguous(), w, out=y)  # wrong K is caught before the call
    L = ops.lib()
    rc = L.w4a16_mm(x.data_ptr() + 2, w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), y.data_ptr(),
                    2, N, K, None)
    assert rc == ops.ERR_ALIGN
    monkeypatch.setenv("W4A16_FAULT", "launch")
    L.w4a16_debug_reload_env()
    try:
        with pytest.raises(ops.W4A16Error):
            ops.mm(x, w, out=y)
    finally:
        monkeypatch.delenv("W4A16_FAULT")
        L.w4a16_debug_reload_env()
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)
    ops.mm(x, w, out=y)  # the context is still usable
    torch.cuda.synchronize()
    assert not torch.all(y == 5.0)
