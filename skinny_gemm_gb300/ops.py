"""Python binding of libw4a16.so: argument marshalling only.

Every computation runs in the library's CUDA kernels.  PyTorch supplies the
device memory, the current CUDA stream and the output allocation; there is
no CPU or PyTorch fallback, and a missing or unbuildable library raises.

Names follow the C ABI in ``include/w4a16.h``: ``mm``, ``mm_group``,
``mm_id``, ``unpack``, ``dequant``, ``get_plan``, ``device_status``; and in
``include/stq1.h`` for the STQ1_0 ternary format: ``stq1_mm``,
``stq1_mm_id``, ``stq1_get_rows``, ``stq1_get_plan`` over an ``STQ1Matrix``
(repacked on the device by ``stq1_pack``).
"""
from __future__ import annotations

import ctypes
import threading
from dataclasses import dataclass

import torch

from . import _build

GROUP = 64

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_EXPERTS, ERR_CUDA, ERR_KERNEL, ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6, -7
KERNELS = {"auto": 0, "simt": 1, "tc": 2, "vanilla": 3, "tc_stream": 4, "tc_tile": 5, "tc_prefill": 6}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}
DEVICE_BAD_ID = 1

EXPORTS = ("w4a16_mm", "w4a16_mm_ws", "w4a16_mm_g", "w4a16_workspace_bytes", "w4a16_mm_kernel", "w4a16_mm_noalloc", "w4a16_mm_group", "w4a16_mm_argmax", "w4a16_embed", "w4a16_expand_groups",
           "w4a16_mm_id", "w4a16_mm_id_kernel", "w4a16_unpack", "w4a16_dequant", "w4a16_get_plan", "w4a16_device_status", "w4a16_last_error",
           "w4a16_debug_reload_env", "w4a16_version",
           "stq1_packed_bytes", "stq1_pack", "stq1_mm", "stq1_mm_id", "stq1_get_rows", "stq1_get_plan")
MAX_GROUP = 8
STQ1_BLOCK_WEIGHTS, STQ1_BLOCK_BYTES = 256, 42


class W4A16Error(RuntimeError):
    """A library call failed; ``status`` is the w4a16_status code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"w4a16 status {status}: {message}")
        self.status = status


class W4A16ValueError(W4A16Error, ValueError):
    pass


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("ksplit", ctypes.c_int), ("slice_k", ctypes.c_int),
                ("rows_per_tile", ctypes.c_int), ("units", ctypes.c_int), ("threads", ctypes.c_int),
                ("grid_x", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("workspace_bytes", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel"] = KERNEL_NAMES.get(self.kernel, self.kernel)
        return d


class Stq1Plan(ctypes.Structure):
    _fields_ = [("ksplit", ctypes.c_int), ("blocks_per_slice", ctypes.c_int), ("rows_per_pass", ctypes.c_int)]


class Item(ctypes.Structure):
    """w4a16_mm_item: one projection of a w4a16_mm_group call (device pointers)."""
    _fields_ = [("x", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int)]


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def library_path() -> str:
    return _build.CUDA_LIB


def lib() -> ctypes.CDLL:
    """Open libw4a16.so (building it in-tree if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build_cuda()
            L = ctypes.CDLL(path)
            P, i, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.w4a16_mm.argtypes = [P, P, P, P, P, i, i, i, P]
            L.w4a16_mm_ws.argtypes = [P, P, P, P, P, i, i, i, P, z, P]
            L.w4a16_mm_g.argtypes = [P, P, P, P, P, i, i, i, i, P, z, P]
            L.w4a16_workspace_bytes.argtypes = [i, i]
            L.w4a16_workspace_bytes.restype = z
            L.w4a16_mm_kernel.argtypes = [P, P, P, P, P, i, i, i, i, P]
            L.w4a16_mm_noalloc.argtypes = [P, P, P, P, P, i, i, i, P]
            L.w4a16_mm_group.argtypes = [ctypes.POINTER(Item), i, i, i, P]
            L.w4a16_mm_argmax.argtypes = [P, P, P, P, P, P, i, i, i, P, z, P]
            L.w4a16_embed.argtypes = [P, P, P, P, P, i, i, i, P]
            L.w4a16_expand_groups.argtypes = [P, P, i, i, i, P]
            L.w4a16_mm_id.argtypes = [P, P, P, P, P, P, i, i, i, i, P]
            L.w4a16_mm_id_kernel.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P]
            L.w4a16_unpack.argtypes = [P, P, i, i, P]
            L.w4a16_dequant.argtypes = [P, P, P, P, i, i, P]
            L.w4a16_get_plan.argtypes = [i, i, i, ctypes.POINTER(Plan)]
            L.w4a16_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
            L.stq1_packed_bytes.argtypes = [i, i]
            L.stq1_packed_bytes.restype = ctypes.c_size_t
            L.stq1_pack.argtypes = [P, P, i, i, P]
            L.stq1_mm.argtypes = [P, P, P, i, i, i, P]
            L.stq1_mm_id.argtypes = [P, P, P, P, i, i, i, i, P]
            L.stq1_get_rows.argtypes = [P, P, P, i, i, i, P]
            L.stq1_get_plan.argtypes = [i, i, ctypes.POINTER(Stq1Plan)]
            for f in ("w4a16_mm", "w4a16_mm_ws", "w4a16_mm_g", "w4a16_mm_kernel", "w4a16_mm_noalloc", "w4a16_mm_group", "w4a16_mm_argmax",
                      "w4a16_embed", "w4a16_expand_groups", "w4a16_mm_id", "w4a16_mm_id_kernel", "w4a16_unpack", "w4a16_dequant",
                      "w4a16_get_plan", "w4a16_device_status", "stq1_pack", "stq1_mm", "stq1_mm_id", "stq1_get_rows",
                      "stq1_get_plan"):
                getattr(L, f).restype = ctypes.c_int
            L.w4a16_last_error.restype = ctypes.c_char_p
            L.w4a16_version.restype = ctypes.c_char_p
            L.w4a16_debug_reload_env.restype = None
            _lib = L
    return _lib


def _raise(rc: int) -> None:
    if rc == OK:
        return
    msg = (lib().w4a16_last_error() or b"").decode()
    if rc in (ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_EXPERTS, ERR_KERNEL):
        raise W4A16ValueError(rc, msg)
    raise W4A16Error(rc, msg)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev_tensor(t: torch.Tensor, dtype: torch.dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---- workspaces (include/w4a16.h "Workspace") --------------------------------------------
#
# The library allocates nothing; this binding is its caller and owns the
# workspaces: one zeroed block per (device, stream), made with torch on the
# first call on that stream outside graph capture (a call captured before
# one exists runs without a workspace, which gives the same bits).

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace_bytes(N: int, K: int) -> int:
    return int(lib().w4a16_workspace_bytes(N, K))


def _capturing() -> bool:
    try:
        return bool(torch.cuda.is_current_stream_capturing())
    except Exception:
        return False


def workspace(stream=None, create: bool = True):
    """The zeroed workspace of the current device and `stream` (uint8 tensor),
    or None when there is none yet and one cannot be made now."""
    s = stream if stream is not None else torch.cuda.current_stream()
    key = (s.device.index if s.device.index is not None else torch.cuda.current_device(), int(s.cuda_stream))
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None and create and not _capturing():
            n = int(lib().w4a16_workspace_bytes(512, 512))
            ws = torch.zeros(n, dtype=torch.uint8, device=f"cuda:{key[0]}")
            torch.cuda.current_stream(ws.device).synchronize()
            _ws_cache[key] = ws
        return ws


def _ws_args(ws):
    if ws is None:
        return None, 0
    _dev_tensor(ws, torch.uint8, "workspace")
    return ws.data_ptr(), ws.numel()


def _g64(w, what: str) -> None:
    if w.group != GROUP:
        raise ValueError(f"{what} takes group-64 tables; expand group {w.group} with W4Matrix.from_group")


def _kernel_id(kernel) -> int:
    if kernel is None:
        return 0
    if isinstance(kernel, str):
        if kernel not in KERNELS:
            raise ValueError(f"unknown kernel {kernel!r}; one of {sorted(KERNELS)}")
        return KERNELS[kernel]
    return int(kernel)


@dataclass
class W4Matrix:
    """Packed W4A16 weights on the GPU.

    Wq: int32 [.., N, K/8] (bit pattern of the uint32 words, eight codes each,
    low nibble first); scales, biases: bfloat16 [.., N, K/group] (group 64,
    or 128 for a single matrix read natively by ``mm``).  With E > 1 the
    leading dimension stacks E experts.
    """

    Wq: torch.Tensor
    scales: torch.Tensor
    biases: torch.Tensor
    N: int
    K: int
    E: int = 1
    group: int = GROUP

    def __post_init__(self):
        lead = () if self.E == 1 else (self.E,)
        if self.group not in (GROUP, 128) or (self.group != GROUP and self.E != 1):
            raise ValueError(f"group {self.group}: 64, or 128 for a single matrix")
        if tuple(self.Wq.shape) != lead + (self.N, self.K // 8):
            raise ValueError(f"Wq shape {tuple(self.Wq.shape)} does not match N={self.N}, K={self.K}, E={self.E}")
        for name in ("scales", "biases"):
            t = getattr(self, name)
            if tuple(t.shape) != lead + (self.N, self.K // self.group):
                raise ValueError(f"{name} shape {tuple(t.shape)} does not match N={self.N}, K={self.K}, "
                                 f"group={self.group}")
        _dev_tensor(self.Wq, torch.int32, "Wq")
        _dev_tensor(self.scales, torch.bfloat16, "scales")
        _dev_tensor(self.biases, torch.bfloat16, "biases")

    @classmethod
    def from_host(cls, host, device="cuda") -> "W4Matrix":
        """From numpy arrays (``synth.HostW4``: uint32 codes, bf16 bit patterns)."""
        wq = torch.from_numpy(host.Wq.view("int32")).to(device)
        s = torch.from_numpy(host.scales.view("int16")).view(torch.bfloat16).to(device)
        b = torch.from_numpy(host.biases.view("int16")).view(torch.bfloat16).to(device)
        return cls(wq, s, b, host.N, host.K, host.E)

    @classmethod
    def from_group(cls, Wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, N: int, K: int,
                   group: int, stream=None) -> "W4Matrix":
        """A table quantized with `group` codes per scale and bias (a multiple
        of 64, e.g. the book's 128): scales/biases bf16 [N][K/group] expanded
        once on the device through ``w4a16_expand_groups``.  The stream is
        synchronised after the expansion: the tensor-core calls may fetch
        weights before earlier kernels on their stream finish (the
        overlapped-launch contract of include/w4a16.h)."""
        _dev_tensor(scales, torch.bfloat16, "scales")
        _dev_tensor(biases, torch.bfloat16, "biases")
        if scales.numel() != N * (K // group) or biases.numel() != N * (K // group):
            raise ValueError(f"scales and biases must hold N * K / group = {N * (K // group)} values")
        out = []
        for t in (scales, biases):
            d = torch.empty(N, K // GROUP, dtype=torch.bfloat16, device=t.device)
            _raise(lib().w4a16_expand_groups(t.data_ptr(), d.data_ptr(), N, K, group, _stream_ptr(stream)))
            out.append(d)
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
        return cls(Wq, out[0], out[1], N, K)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.Wq, self.scales, self.biases))


def mm(x: torch.Tensor, w: W4Matrix, out: torch.Tensor | None = None, kernel=None, stream=None,
       workspace="auto") -> torch.Tensor:
    """y[..., N] = x[..., K] W^T (leading dims flatten into M) through
    ``w4a16_mm_ws`` with this stream's workspace (``workspace="auto"``), a
    given uint8 workspace tensor, or ``w4a16_mm`` (``workspace=None``); an
    explicit ``kernel`` goes through ``w4a16_mm_kernel`` without one."""
    if w.E != 1:
        raise ValueError("mm takes a single matrix; use mm_id for stacked experts")
    _dev_tensor(x, torch.bfloat16, "x")
    if x.shape[-1] != w.K:
        raise ValueError(f"x has K={x.shape[-1]}, weights have K={w.K}")
    if w.group != GROUP and kernel not in (None, "auto", 0):
        raise ValueError("group-128 tables run on their own kernel; no kernel selection")
    M = x.numel() // w.K
    if out is None:
        out = torch.empty(*x.shape[:-1], w.N, dtype=torch.bfloat16, device=x.device)
    _dev_tensor(out, torch.bfloat16, "out")
    if out.numel() != M * w.N:
        raise ValueError("out has the wrong number of elements")
    L = lib()
    k = _kernel_id(kernel)
    args = (x.data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), out.data_ptr(), M, w.N, w.K)
    if w.group != GROUP:
        ws = globals()["workspace"](stream) if isinstance(workspace, str) else workspace
        rc = L.w4a16_mm_g(*args, w.group, *_ws_args(ws), _stream_ptr(stream))
    elif k != 0:
        rc = L.w4a16_mm_kernel(*args, k, _stream_ptr(stream))
    else:
        ws = globals()["workspace"](stream) if isinstance(workspace, str) else workspace
        if ws is None:
            rc = L.w4a16_mm(*args, _stream_ptr(stream))
        else:
            rc = L.w4a16_mm_ws(*args, *_ws_args(ws), _stream_ptr(stream))
    _raise(rc)
    return out


def mm_argmax(x: torch.Tensor, w: W4Matrix, idx: torch.Tensor | None = None, val: torch.Tensor | None = None,
              stream=None, workspace="auto"):
    """(idx, val) through ``w4a16_mm_argmax``: for every row of x (leading dims
    flatten into M) the index of the largest output of ``mm(x, w)`` and that
    output (ties to the smallest index), without writing the outputs.

    idx is int32 [..], val bf16 [..]; pass ``val=False`` to skip the values.
    The call needs a workspace: this stream's (``"auto"``; make one call on
    the stream before capturing it into a CUDA graph) or a given one."""
    _g64(w, "mm_argmax")
    if w.E != 1:
        raise ValueError("mm_argmax takes a single matrix")
    _dev_tensor(x, torch.bfloat16, "x")
    if x.shape[-1] != w.K:
        raise ValueError(f"x has K={x.shape[-1]}, weights have K={w.K}")
    M = x.numel() // w.K
    if idx is None:
        idx = torch.empty(x.shape[:-1], dtype=torch.int32, device=x.device)
    _dev_tensor(idx, torch.int32, "idx")
    if idx.numel() != M:
        raise ValueError("idx must have one element per row")
    if val is None:
        val = torch.empty(x.shape[:-1], dtype=torch.bfloat16, device=x.device)
    if val is not False:
        _dev_tensor(val, torch.bfloat16, "val")
        if val.numel() != M:
            raise ValueError("val must have one element per row")
    vp = val.data_ptr() if val is not False else None
    ws = globals()["workspace"](stream) if isinstance(workspace, str) else workspace
    if ws is None and M > 0:
        raise ValueError("mm_argmax needs a workspace: call it once on this stream before graph capture, "
                         "or pass workspace=")
    rc = lib().w4a16_mm_argmax(x.data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), idx.data_ptr(),
                               vp, M, w.N, w.K, *_ws_args(ws), _stream_ptr(stream))
    _raise(rc)
    return idx, (val if val is not False else None)


def embed(ids: torch.Tensor, w: W4Matrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rows ids of the packed table w (N rows of width K), dequantized to bf16
    [..., K] through ``w4a16_embed``; ids int32 on the device."""
    _g64(w, "embed")
    if w.E != 1:
        raise ValueError("embed takes a single table")
    _dev_tensor(ids, torch.int32, "ids")
    T = ids.numel()
    if out is None:
        out = torch.empty(*ids.shape, w.K, dtype=torch.bfloat16, device=ids.device)
    _dev_tensor(out, torch.bfloat16, "out")
    if out.numel() != T * w.K:
        raise ValueError("out has the wrong number of elements")
    rc = lib().w4a16_embed(w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), ids.data_ptr(), out.data_ptr(),
                           T, w.N, w.K, _stream_ptr(stream))
    _raise(rc)
    return out


def mm_group(xs, ws, outs=None, stream=None) -> list:
    """[mm(x, w) for x, w in zip(xs, ws)] through one ``w4a16_mm_group`` call.

    The projections must share K and the number of activation rows M; each
    result equals ``mm(x, w)`` bit for bit."""
    xs, ws = list(xs), list(ws)
    if not 1 <= len(xs) == len(ws) <= MAX_GROUP:
        raise ValueError(f"need 1..{MAX_GROUP} (x, w) pairs")
    K = ws[0].K
    M = xs[0].numel() // K if K else 0
    if outs is None:
        outs = [torch.empty(*x.shape[:-1], w.N, dtype=torch.bfloat16, device=x.device) for x, w in zip(xs, ws)]
    items = (Item * len(xs))()
    for i, (x, w, y) in enumerate(zip(xs, ws, outs)):
        if w.E != 1:
            raise ValueError("mm_group takes single matrices")
        _g64(w, "mm_group")
        _dev_tensor(x, torch.bfloat16, "x")
        _dev_tensor(y, torch.bfloat16, "out")
        if w.K != K or x.shape[-1] != K or x.numel() != M * K:
            raise ValueError("every item must have the same K and the same number of rows")
        if y.numel() != M * w.N:
            raise ValueError("out has the wrong number of elements")
        items[i] = Item(x.data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), y.data_ptr(), w.N)
    _raise(lib().w4a16_mm_group(items, len(xs), M, K, _stream_ptr(stream)))
    return outs


def mm_id(x: torch.Tensor, w: W4Matrix, ids: torch.Tensor, out: torch.Tensor | None = None, kernel=None,
          stream=None) -> torch.Tensor:
    """y[t] = W[ids[t]] x[t] through ``w4a16_mm_id``; x [T, K], ids int32 [T] on the GPU."""
    _g64(w, "mm_id")
    _dev_tensor(x, torch.bfloat16, "x")
    _dev_tensor(ids, torch.int32, "ids")
    if x.dim() != 2 or x.shape[1] != w.K:
        raise ValueError("x must be [T, K]")
    T = x.shape[0]
    if ids.numel() != T:
        raise ValueError("ids must hold one expert id per token")
    if out is None:
        out = torch.empty(T, w.N, dtype=torch.bfloat16, device=x.device)
    _dev_tensor(out, torch.bfloat16, "out")
    L = lib()
    rc = L.w4a16_mm_id_kernel(x.data_ptr(), w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(),
                              ids.data_ptr(), out.data_ptr(), T, w.N, w.K, w.E, _kernel_id(kernel),
                              _stream_ptr(stream))
    _raise(rc)
    return out


def unpack(w: W4Matrix, stream=None) -> torch.Tensor:
    """Codes q[N][K] as uint8 through ``w4a16_unpack`` (bit-exact debug path)."""
    q = torch.empty(w.N, w.K, dtype=torch.uint8, device=w.Wq.device)
    _raise(lib().w4a16_unpack(w.Wq.data_ptr(), q.data_ptr(), w.N, w.K, _stream_ptr(stream)))
    return q


def dequant(w: W4Matrix, stream=None) -> torch.Tensor:
    """fp32 weights fma(q, s, b) [N][K] through ``w4a16_dequant``."""
    _g64(w, "dequant")
    out = torch.empty(w.N, w.K, dtype=torch.float32, device=w.Wq.device)
    _raise(lib().w4a16_dequant(w.Wq.data_ptr(), w.scales.data_ptr(), w.biases.data_ptr(), out.data_ptr(),
                               w.N, w.K, _stream_ptr(stream)))
    return out


def get_plan(N: int, K: int, kernel=None) -> dict:
    p = Plan()
    _raise(lib().w4a16_get_plan(N, K, _kernel_id(kernel), ctypes.byref(p)))
    return p.as_dict()


def device_status(stream=None) -> int:
    """Synchronise and return (then clear) the device flags; raises on CUDA errors only."""
    flags = ctypes.c_int(0)
    rc = lib().w4a16_device_status(_stream_ptr(stream), ctypes.byref(flags))
    if rc not in (OK, ERR_DEVICE):
        _raise(rc)
    return flags.value


# ---- STQ1_0 ternary matrices (include/stq1.h) -------------------------------------------

@dataclass
class STQ1Matrix:
    """An STQ1_0 matrix (or E stacked experts) repacked on the GPU for the
    stq1 kernels: ``packed`` uint8 [E * stq1_packed_bytes(N, K)]."""

    packed: torch.Tensor
    N: int
    K: int
    E: int = 1

    @classmethod
    def from_blocks(cls, blocks: torch.Tensor, N: int, K: int, E: int = 1, stream=None) -> "STQ1Matrix":
        """From the page's 42-byte blocks, uint8 [.., N, K/256, 42] on the GPU."""
        _dev_tensor(blocks, torch.uint8, "blocks")
        per = stq1_packed_bytes(N, K)
        if per == 0:
            raise ValueError(f"STQ1_0 needs N >= 1 and K a multiple of 256 in 256..32768 (N={N}, K={K})")
        if blocks.numel() != E * N * (K // STQ1_BLOCK_WEIGHTS) * STQ1_BLOCK_BYTES:
            raise ValueError("blocks must hold E * N * K/256 blocks of 42 bytes")
        packed = torch.empty(E * per, dtype=torch.uint8, device=blocks.device)
        src = blocks.reshape(E, -1)
        for e in range(E):
            _raise(lib().stq1_pack(src[e].data_ptr(), packed.data_ptr() + e * per, N, K, _stream_ptr(stream)))
        return cls(packed, N, K, E)

    @classmethod
    def from_host(cls, blocks, N: int, K: int, E: int = 1, device="cuda") -> "STQ1Matrix":
        """From a numpy uint8 array of blocks (``synth.make_stq1``)."""
        return cls.from_blocks(torch.from_numpy(blocks.reshape(-1).copy()).to(device), N, K, E)

    @property
    def nbytes(self) -> int:
        """Bytes of the weights in the page's format (42 per 256 weights)."""
        return self.E * self.N * (self.K // STQ1_BLOCK_WEIGHTS) * STQ1_BLOCK_BYTES


def stq1_packed_bytes(N: int, K: int) -> int:
    return int(lib().stq1_packed_bytes(N, K))


def stq1_mm(x: torch.Tensor, w: STQ1Matrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[..., N] = x[..., K] W^T (float32) through ``stq1_mm``."""
    if w.E != 1:
        raise ValueError("stq1_mm takes a single matrix; use stq1_mm_id for stacked experts")
    _dev_tensor(x, torch.float32, "x")
    if x.shape[-1] != w.K:
        raise ValueError(f"x has K={x.shape[-1]}, weights have K={w.K}")
    M = x.numel() // w.K
    if out is None:
        out = torch.empty(*x.shape[:-1], w.N, dtype=torch.float32, device=x.device)
    _dev_tensor(out, torch.float32, "out")
    if out.numel() != M * w.N:
        raise ValueError("out has the wrong number of elements")
    _raise(lib().stq1_mm(x.data_ptr(), w.packed.data_ptr(), out.data_ptr(), M, w.N, w.K, _stream_ptr(stream)))
    return out


def stq1_mm_id(x: torch.Tensor, w: STQ1Matrix, ids: torch.Tensor, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """y[t] = W[ids[t]] x[t] (float32) through ``stq1_mm_id``; x [T, K], ids int32 [T]."""
    _dev_tensor(x, torch.float32, "x")
    _dev_tensor(ids, torch.int32, "ids")
    if x.dim() != 2 or x.shape[1] != w.K:
        raise ValueError("x must be [T, K]")
    T = x.shape[0]
    if ids.numel() != T:
        raise ValueError("ids must hold one expert id per token")
    if out is None:
        out = torch.empty(T, w.N, dtype=torch.float32, device=x.device)
    _dev_tensor(out, torch.float32, "out")
    _raise(lib().stq1_mm_id(x.data_ptr(), w.packed.data_ptr(), ids.data_ptr(), out.data_ptr(), T, w.N, w.K, w.E,
                            _stream_ptr(stream)))
    return out


def stq1_get_rows(ids: torch.Tensor, w: STQ1Matrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rows ids of W as float32 [..., K] through ``stq1_get_rows``."""
    if w.E != 1:
        raise ValueError("stq1_get_rows takes a single matrix")
    _dev_tensor(ids, torch.int32, "ids")
    T = ids.numel()
    if out is None:
        out = torch.empty(*ids.shape, w.K, dtype=torch.float32, device=ids.device)
    _dev_tensor(out, torch.float32, "out")
    if out.numel() != T * w.K:
        raise ValueError("out has the wrong number of elements")
    _raise(lib().stq1_get_rows(w.packed.data_ptr(), ids.data_ptr(), out.data_ptr(), T, w.N, w.K,
                               _stream_ptr(stream)))
    return out


def stq1_get_plan(N: int, K: int) -> dict:
    p = Stq1Plan()
    _raise(lib().stq1_get_plan(N, K, ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in p._fields_}


def version() -> str:
    return lib().w4a16_version().decode()
