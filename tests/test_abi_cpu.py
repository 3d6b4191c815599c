"""The C-ABI library on the host: it loads, exports what include/*.h declares,
and rejects bad arguments before any launch (no GPU needed).

Fake device pointers below are never dereferenced: every call here fails in
host validation (or is an M == 0 no-op) before the library touches CUDA.
"""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from skinny_gemm_gb300 import _build, ops, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DECL = re.compile(r"^\s*(?:int|void|size_t|const char\s*\*)\s+(w4a16_\w+)\s*\(", re.M)
STQ1_DECL = re.compile(r"^\s*(?:int|size_t)\s+(stq1_\w+)\s*\(", re.M)

P = 0x10000  # 16-byte-aligned fake address


def _declared(header: str) -> list[str]:
    return DECL.findall(open(os.path.join(ROOT, "include", header)).read())


def _exported(path: str) -> set[str]:
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_every_declared_symbol_is_exported():
    headers = sorted(os.path.basename(h) for h in glob.glob(os.path.join(ROOT, "include", "*.h")))
    assert headers == ["stq1.h", "w4a16.h", "w4a16_synth.h"]
    cuda_syms = _exported(_build.build_cuda())
    decl = _declared("w4a16.h")
    assert len(decl) >= 10
    missing = [s for s in decl if s not in cuda_syms]
    assert not missing, f"declared but not exported by libw4a16.so: {missing}"
    decl = STQ1_DECL.findall(open(os.path.join(ROOT, "include", "stq1.h")).read())
    assert len(decl) == 6
    missing = [s for s in decl if s not in cuda_syms]
    assert not missing, f"declared in stq1.h but not exported by libw4a16.so: {missing}"
    synth_syms = _exported(_build.build_synth())
    decl = _declared("w4a16_synth.h")
    assert len(decl) == 9
    assert not [s for s in decl if s not in synth_syms]
    # the binding names exactly the exported C calls
    assert set(ops.EXPORTS) <= cuda_syms


@pytest.fixture()
def L(monkeypatch):
    monkeypatch.delenv("W4A16_FAULT", raising=False)
    monkeypatch.delenv("W4A16_FORCE_KERNEL", raising=False)
    lib = ops.lib()
    lib.w4a16_debug_reload_env()
    yield lib
    monkeypatch.delenv("W4A16_FAULT", raising=False)
    lib.w4a16_debug_reload_env()


def _mm(L, x=P, w=P, s=P, b=P, y=P, M=1, N=256, K=512, kernel=None):
    if kernel is None:
        return L.w4a16_mm(x, w, s, b, y, M, N, K, None)
    return L.w4a16_mm_kernel(x, w, s, b, y, M, N, K, kernel, None)


def _err(L) -> str:
    return L.w4a16_last_error().decode()


def test_shape_errors(L):
    assert _mm(L, K=100) == ops.ERR_SHAPE and "multiple of 64" in _err(L)
    assert _mm(L, K=0) == ops.ERR_SHAPE
    assert _mm(L, K=-64) == ops.ERR_SHAPE
    assert _mm(L, N=0) == ops.ERR_SHAPE
    assert _mm(L, N=-3) == ops.ERR_SHAPE
    assert _mm(L, M=-1) == ops.ERR_SHAPE


def test_null_and_alignment_errors(L):
    assert _mm(L, x=None) == ops.ERR_NULL
    assert _mm(L, y=None) == ops.ERR_NULL
    assert _mm(L, x=P + 8) == ops.ERR_ALIGN
    assert _mm(L, w=P + 4) == ops.ERR_ALIGN
    assert _mm(L, s=P + 1) == ops.ERR_ALIGN
    assert _mm(L, b=P + 4) == ops.ERR_ALIGN
    assert _mm(L, y=P + 1) == ops.ERR_ALIGN
    assert "16-byte" in (_mm(L, x=P + 2) and _err(L))


def test_empty_batch_is_a_noop_without_cuda(L):
    # M == 0 returns before any CUDA call, so it succeeds even with no GPU
    assert _mm(L, x=None, w=None, s=None, b=None, y=None, M=0) == ops.OK
    assert L.w4a16_mm_id(None, None, None, None, None, None, 0, 64, 64, 4, None) == ops.OK


def test_unknown_kernel(L):
    assert _mm(L, kernel=42) == ops.ERR_KERNEL


def test_mm_id_errors(L):
    assert L.w4a16_mm_id(P, P, P, P, P, P, 8, 64, 64, 0, None) == ops.ERR_EXPERTS
    assert L.w4a16_mm_id(P, P, P, P, P, P, -1, 64, 64, 8, None) == ops.ERR_EXPERTS
    assert L.w4a16_mm_id(P, P, P, P, P, P, 8, 64, 96, 8, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_id(P, P, P, P, P + 2, P, 8, 64, 64, 8, None) == ops.ERR_ALIGN
    assert L.w4a16_mm_id(P, P, P, P, None, P, 8, 64, 64, 8, None) == ops.ERR_NULL
    # K % 512 != 0: the routed tile kernel is refused before anything runs
    assert L.w4a16_mm_id_kernel(P, P, P, P, P, P, 8, 64, 576, 8, ops.KERNELS["tc_tile"], None) == ops.ERR_KERNEL
    assert L.w4a16_mm_id_kernel(P, P, P, P, P, P, 0, 64, 576, 8, ops.KERNELS["tc_tile"], None) == ops.ERR_KERNEL


def test_mm_argmax_errors(L):
    """Fail-closed checks of w4a16_mm_argmax, all before any device call."""
    f = L.w4a16_mm_argmax
    WS, NB = 0x100000, L.w4a16_workspace_bytes(64, 512)
    assert f(P, P, P, P, P, P, 0, 64, 512, None, 0, None) == ops.OK          # M == 0: no-op
    assert f(P, P, P, P, P, None, -1, 64, 512, WS, NB, None) == ops.ERR_SHAPE
    assert f(P, P, P, P, P, P, 1, 64, 96, WS, NB, None) == ops.ERR_SHAPE    # K % 64
    assert f(P, P, P, P, None, P, 1, 64, 512, WS, NB, None) == ops.ERR_NULL  # idx
    assert f(P + 8, P, P, P, P, P, 1, 64, 512, WS, NB, None) == ops.ERR_ALIGN
    assert f(P, P, P, P, P + 2, P, 1, 64, 512, WS, NB, None) == ops.ERR_ALIGN  # idx 4-byte
    assert f(P, P, P, P, P, P + 1, 1, 64, 512, WS, NB, None) == ops.ERR_ALIGN  # val 2-byte
    assert f(P, P, P, P, P, P, 1, 64, 512, None, 0, None) == ops.ERR_NULL    # no workspace
    assert f(P, P, P, P, P, P, 1, 64, 512, WS, NB - 1, None) == ops.ERR_SHAPE  # too small
    assert f(P, P, P, P, P, P, 1, 64, 512, WS + 16, NB, None) == ops.ERR_ALIGN  # 256-byte alignment
    assert f(P, P, P, P, P, P, 1, 64, 448, WS, NB, None) == ops.ERR_KERNEL   # K % 512 == 0 only


def test_workspace_bytes_and_mm_ws_errors(L):
    """The workspace query and w4a16_mm_ws's fail-closed checks."""
    nb = L.w4a16_workspace_bytes(262144, 2560)
    assert nb == 5013504  # 32 KiB counters + 4864 KiB fp32 partials, every shape
    assert L.w4a16_workspace_bytes(16384, 16384) == nb
    assert L.w4a16_workspace_bytes(256, 448) == nb    # K % 512 != 0: tensor cores, padded K
    assert L.w4a16_workspace_bytes(0, 512) == 0
    assert L.w4a16_workspace_bytes(64, 96) == 0
    f = L.w4a16_mm_ws
    WS = 0x100000
    assert f(P, P, P, P, P, 0, 64, 512, WS, nb, None) == ops.OK            # M == 0: no-op
    assert f(P, P, P, P, P, 1, 64, 512, WS, nb - 256, None) == ops.ERR_SHAPE
    assert f(P, P, P, P, P, 1, 64, 512, WS + 128, nb, None) == ops.ERR_ALIGN
    assert f(P, P, P, P, P, 1, 64, 96, WS, nb, None) == ops.ERR_SHAPE      # K % 64
    assert f(P, P, P, P, None, 1, 64, 512, WS, nb, None) == ops.ERR_NULL
    # the plan reports the workspace the launch shape takes when one is given
    lm = ops.get_plan(262144, 2560)
    assert lm["kernel"] == "tc" and lm["workspace_bytes"] == nb
    assert ops.get_plan(2048, 2560)["workspace_bytes"] == 0   # the tile kernel needs none
    assert ops.get_plan(256, 448)["workspace_bytes"] == 0


def test_embed_errors(L):
    f = L.w4a16_embed
    assert f(P, P, P, P, P, 0, 64, 64, None) == ops.OK                 # T == 0: no-op
    assert f(P, P, P, P, P, -1, 64, 64, None) == ops.ERR_SHAPE
    assert f(P, P, P, P, P, 65536, 64, 64, None) == ops.ERR_SHAPE
    assert f(P, P, P, P, P, 2, 64, 96, None) == ops.ERR_SHAPE           # K % 64
    assert f(P, P, P, None, P, 2, 64, 64, None) == ops.ERR_NULL         # ids
    assert f(P, P, P, P, P + 8, 2, 64, 64, None) == ops.ERR_ALIGN       # out 16-byte
    assert f(P, P, P, P + 2, P, 2, 64, 64, None) == ops.ERR_ALIGN       # ids 4-byte


def test_expand_groups_errors(L):
    f = L.w4a16_expand_groups
    assert f(P, P, 4, 256, 96, None) == ops.ERR_SHAPE     # not a multiple of 64
    assert f(P, P, 4, 384, 256, None) == ops.ERR_SHAPE    # does not divide K
    assert f(P, P, 4, 96, 128, None) == ops.ERR_SHAPE     # K % 64
    assert f(None, P, 4, 256, 128, None) == ops.ERR_NULL
    assert f(P + 1, P, 4, 256, 128, None) == ops.ERR_ALIGN


def test_debug_entry_point_errors(L):
    assert L.w4a16_unpack(P, P, 4, 12, None) == ops.ERR_SHAPE
    assert L.w4a16_unpack(None, P, 4, 64, None) == ops.ERR_NULL
    assert L.w4a16_dequant(P, P, P, P + 4, 4, 64, None) == ops.ERR_ALIGN
    assert L.w4a16_dequant(P, P, P, P, 4, 32, None) == ops.ERR_SHAPE


def test_injected_faults(L, monkeypatch):
    monkeypatch.setenv("W4A16_FAULT", "validate")
    L.w4a16_debug_reload_env()
    assert _mm(L) == ops.ERR_SHAPE and "injected" in _err(L)
    assert L.w4a16_mm_id(P, P, P, P, P, P, 8, 64, 64, 8, None) == ops.ERR_SHAPE
    monkeypatch.setenv("W4A16_FAULT", "launch")
    L.w4a16_debug_reload_env()
    assert _mm(L) == ops.ERR_CUDA and "injected launch" in _err(L)
    # arguments are still validated first
    assert _mm(L, K=65) == ops.ERR_SHAPE


def test_plans_depend_on_shape_only_and_fill_the_gpu(L):
    shapes = [(256, 512), (2048, 2560), (512, 2560), (2560, 2048), (10240, 2560), (2560, 10240),
              (12288, 1536), (1536, 12288), (262144, 1536), (262144, 2560), (16384, 16384), (6144, 2048)]
    for N, K in shapes:
        for kern in ("auto", "simt", "tc", "vanilla"):
            p = ops.get_plan(N, K, kern)
            assert p["units"] * p["rows_per_tile"] >= N or p["kernel"] == "tc"
            assert p["ksplit"] * p["slice_k"] >= K or p["kernel"] == "simt"
            assert p["ksplit"] >= 1 and p["threads"] % 32 == 0
    with pytest.raises(ValueError):
        ops.get_plan(100, 100)
    # K % 512 != 0 runs on the tensor cores padded to whole 512-code stages
    for K in (64, 192, 768, 2304):
        p = ops.get_plan(100, K)
        assert p["kernel"] == "tc" and p["ksplit"] * p["slice_k"] == -(-K // 512) * 512
        assert ops.get_plan(100, K, "tc")["kernel"] == "tc"
        assert ops.get_plan(100, K, "simt")["kernel"] == "simt"
    assert ops.get_plan(100, 2560)["kernel"] == "tc"
    # the padded slicing of the Gemma-2-sized LM head: 4.5 stages of codes -> five
    p = ops.get_plan(256000, 2304)
    assert p["kernel"] == "tc" and p["ksplit"] * p["slice_k"] == 2560
    # the reduction order is a pure function of (N, K) -- the plan call has no M
    for N, K in shapes:
        a, b = ops.get_plan(N, K), ops.get_plan(N, K)
        assert (a["ksplit"], a["slice_k"]) == (b["ksplit"], b["slice_k"])
        if a["kernel"] == "tc":
            assert (a["ksplit"] - 1) * a["slice_k"] < K <= a["ksplit"] * a["slice_k"]


def test_padded_k_plans(L):
    """K % 512 != 0 runs padded on the tensor cores up to the K whose per-unit
    parameter rows fit in shared memory (5952), on the persistent or the tile
    launch shape; never on the prefill kernel; larger K on the CUDA-core
    family by default."""
    nb = L.w4a16_workspace_bytes(262144, 2560)
    for K in (576, 1152, 2304, 4160, 5952):
        for N in (1, 300, 9216, 256000):
            p = ops.get_plan(N, K)
            assert p["kernel"] == "tc", (N, K, p)
            assert p["ksplit"] * p["slice_k"] >= -(-K // 512) * 512 > (p["ksplit"] - 1) * p["slice_k"]
            assert ops.get_plan(N, K, "tc_stream")["kernel"] == "tc_stream"
            with pytest.raises(ValueError):
                ops.get_plan(N, K, "tc_prefill")
        assert ops.get_plan(300, K, "tc_tile")["kernel"] == "tc_tile"
        assert L.w4a16_workspace_bytes(300, K) == nb
    for K in (6016, 6912, 11008):
        assert ops.get_plan(300, K)["kernel"] == "simt"
        assert L.w4a16_workspace_bytes(300, K) == 0
        with pytest.raises(ValueError):
            ops.get_plan(300, K, "tc")
    # the small and mid shapes take the tile kernel (16-row tiles), the large heads the persistent grid
    assert ops.get_plan(9216, 2304)["rows_per_tile"] == 16
    assert ops.get_plan(256000, 2304)["rows_per_tile"] == 32


def test_split_plans_fit_the_fixed_workspace(L):
    # the persistent kernel's workspace holds 8192 tile counters and 4864 x 32 rows of unit partials
    for K in (512, 1024, 1536, 2048, 2560, 4096, 10240, 12288, 16384, 65536):
        for N in (1, 31, 32, 500, 1621 * 32, 2431 * 32, 2432 * 32, 5000 * 32, 262144):
            p = ops.get_plan(N, K, "tc_stream")
            if p["ksplit"] > 1:
                assert p["units"] * p["rows_per_tile"] <= 4864 * 32, (N, K, p)
                assert p["units"] // p["ksplit"] <= 8192, (N, K, p)


def test_python_layer_rejects_host_tensors():
    import torch
    w = synth.make_weights(0, 64, 64)
    with pytest.raises(ValueError):
        ops.W4Matrix(torch.from_numpy(w.Wq.view("int32")), torch.zeros(64, 1, dtype=torch.bfloat16),
                     torch.zeros(64, 1, dtype=torch.bfloat16), 64, 64)


def test_version_string(L):
    assert "sm_103a" in L.w4a16_version().decode()


def _items(n, N=256, over=None):
    arr = (ops.Item * max(n, 1))()
    for i in range(n):
        f = dict(x=P, Wq=P, scales=P, biases=P, y=P, N=N)
        f.update((over or {}).get(i, {}))
        arr[i] = ops.Item(**f)
    return arr


def test_mm_group_errors(L):
    assert L.w4a16_mm_group(_items(2), 0, 1, 512, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_group(_items(9), 9, 1, 512, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_group(None, 2, 1, 512, None) == ops.ERR_NULL
    assert L.w4a16_mm_group(_items(3), 3, 1, 100, None) == ops.ERR_SHAPE  # K % 64
    assert L.w4a16_mm_group(_items(3, over={2: {"N": 0}}), 3, 1, 512, None) == ops.ERR_SHAPE
    assert L.w4a16_mm_group(_items(3, over={1: {"y": None}}), 3, 1, 512, None) == ops.ERR_NULL
    assert L.w4a16_mm_group(_items(3, over={1: {"x": P + 8}}), 3, 1, 512, None) == ops.ERR_ALIGN
    # M == 0 is a no-op once every item is valid, and items are still checked
    assert L.w4a16_mm_group(_items(3), 3, 0, 512, None) == ops.OK
    assert L.w4a16_mm_group(_items(3, over={0: {"N": -1}}), 3, 0, 512, None) == ops.ERR_SHAPE


def test_stq1_sizes_plans_and_errors(L, monkeypatch):
    assert L.stq1_packed_bytes(16, 256) == 672
    assert L.stq1_packed_bytes(17, 512) == 2 * 2 * 672
    assert L.stq1_packed_bytes(6144, 2048) == 6144 * 8 * 42            # the page's bytes when N % 16 == 0
    for N, K in [(0, 256), (4, 300), (4, 0), (4, 32768 + 256)]:
        assert L.stq1_packed_bytes(N, K) == 0
    plan = ops.Stq1Plan()
    assert L.stq1_get_plan(6144, 2048, ctypes.byref(plan)) == ops.OK
    assert (plan.ksplit, plan.blocks_per_slice, plan.rows_per_pass) == (8, 1, 8)
    assert L.stq1_get_plan(16384, 16384, ctypes.byref(plan)) == ops.OK
    assert (plan.ksplit, plan.blocks_per_slice, plan.rows_per_pass) == (4, 16, 8)
    assert L.stq1_get_plan(16, 256, ctypes.byref(plan)) == ops.OK and plan.ksplit == 1
    assert L.stq1_get_plan(4, 384, ctypes.byref(plan)) == ops.ERR_SHAPE
    assert L.stq1_get_plan(4, 32768, ctypes.byref(plan)) == ops.OK and plan.rows_per_pass == 8
    assert (plan.ksplit, plan.blocks_per_slice) == (8, 16)
    mm, mid, rows, pack = L.stq1_mm, L.stq1_mm_id, L.stq1_get_rows, L.stq1_pack
    assert mm(P, P, P, 0, 64, 512, None) == ops.OK                      # M == 0: no-op
    assert mm(P, P, P, -1, 64, 512, None) == ops.ERR_SHAPE
    assert mm(P, P, P, 1, 64, 320, None) == ops.ERR_SHAPE and "multiple of 256" in _err(L)
    assert mm(P, P, P, 1, 0, 512, None) == ops.ERR_SHAPE
    assert mm(None, P, P, 1, 64, 512, None) == ops.ERR_NULL
    assert mm(P + 4, P, P, 1, 64, 512, None) == ops.ERR_ALIGN
    assert mm(P, P + 8, P, 1, 64, 512, None) == ops.ERR_ALIGN
    assert mm(P, P, P + 2, 1, 64, 512, None) == ops.ERR_ALIGN
    assert mid(P, P, P, P, 0, 64, 512, 8, None) == ops.OK
    assert mid(P, P, P, P, 4, 64, 512, 0, None) == ops.ERR_EXPERTS
    assert mid(P, P, P, P, -1, 64, 512, 8, None) == ops.ERR_EXPERTS
    assert mid(P, P, None, P, 4, 64, 512, 8, None) == ops.ERR_NULL
    assert mid(P, P, P + 2, P, 4, 64, 512, 8, None) == ops.ERR_ALIGN
    assert rows(P, P, P, 0, 64, 512, None) == ops.OK
    assert rows(P, None, P, 3, 64, 512, None) == ops.ERR_NULL
    assert rows(P, P, P, 3, 64, 500, None) == ops.ERR_SHAPE
    assert pack(P + 1, P, 64, 512, None) == ops.ERR_ALIGN                 # blocks 2-byte
    assert pack(P, P + 8, 64, 512, None) == ops.ERR_ALIGN                 # packed 16-byte
    assert pack(P, P, 64, 128, None) == ops.ERR_SHAPE
    monkeypatch.setenv("W4A16_FAULT", "validate")
    L.w4a16_debug_reload_env()
    assert mm(P, P, P, 1, 64, 512, None) == ops.ERR_SHAPE and "injected" in _err(L)


def test_stq1_plans_depend_on_shape_only():
    """The K split and the rows per pass are functions of (N, K): 256 weight
    rows per CTA, K over a cluster of at most 8 CTAs and at most one slice
    per block, as many slices as keep the grid within 256 CTAs (one wave at
    two per SM), each slice non-empty; eight activation rows per pass."""
    L = ops.lib()
    for N, K in [(16, 256), (6144, 2048), (16384, 16384), (2048, 2560), (300, 4096), (262144, 1536),
                 (40, 32768), (7, 8192), (1000, 12288)]:
        plans = []
        for _ in range(2):
            p = ops.Stq1Plan()
            assert L.stq1_get_plan(N, K, ctypes.byref(p)) == ops.OK
            plans.append((p.ksplit, p.blocks_per_slice, p.rows_per_pass))
        ks, bps, rows = plans[0]
        assert plans[0] == plans[1]
        nb, groups = K // 256, -(-N // 256)
        assert 1 <= ks <= min(8, nb) and (ks - 1) * bps < nb <= ks * bps, (N, K, ks, bps)
        want = max(1, min(8, nb, 256 // groups))
        assert bps == -(-nb // want), (N, K, ks, bps)
        assert rows == 8


def test_stq1_python_layer_checks_before_any_launch():
    """Host tensors, wrong dtypes and wrong block counts are refused in Python;
    shapes the library rejects raise its ValueError (no device needed)."""
    import torch
    blocks = torch.zeros(4 * 2 * 42, dtype=torch.uint8)
    with pytest.raises(ValueError):
        ops.STQ1Matrix.from_blocks(blocks, 4, 512)                       # a host tensor
    with pytest.raises(ValueError):
        ops.STQ1Matrix.from_blocks(blocks, 4, 300)                       # K % 256
    w = ops.STQ1Matrix(torch.zeros(ops.stq1_packed_bytes(4, 512), dtype=torch.uint8), 4, 512)
    with pytest.raises(ValueError):
        ops.stq1_mm(torch.zeros(1, 512, dtype=torch.bfloat16), w)        # not float32 / not on the GPU
    with pytest.raises(ValueError):
        ops.stq1_get_rows(torch.zeros(3, dtype=torch.int64), w)          # ids must be int32
    with pytest.raises(ops.W4A16ValueError):
        ops.stq1_get_plan(4, 384)
    assert ops.stq1_get_plan(6144, 2048) == {"ksplit": 8, "blocks_per_slice": 1, "rows_per_pass": 8}


def test_mm_g_errors(L):
    """w4a16_mm_g: group 64 is w4a16_mm_ws; group 128 needs K % 512 == 0 up
    to 8192 and 16-byte aligned tables; everything fails before a launch."""
    f = L.w4a16_mm_g
    assert f(P, P, P, P, P, 0, 64, 512, 128, None, 0, None) == ops.OK            # M == 0
    assert f(P, P, P, P, P, 1, 64, 512, 96, None, 0, None) == ops.ERR_SHAPE      # group
    assert f(P, P, P, P, P, 1, 64, 768, 128, None, 0, None) == ops.ERR_SHAPE     # K % 512
    assert f(P, P, P, P, P, 1, 64, 8704, 128, None, 0, None) == ops.ERR_SHAPE    # K > 8192
    assert f(P, P, P + 8, P, P, 1, 64, 512, 128, None, 0, None) == ops.ERR_ALIGN  # scales 16-byte
    assert f(P, P, P, P, None, 1, 64, 512, 128, None, 0, None) == ops.ERR_NULL
    assert f(P, P, P, P, P, 1, 64, 512, 128, 0x100000, 100, None) == ops.ERR_SHAPE  # workspace too small
