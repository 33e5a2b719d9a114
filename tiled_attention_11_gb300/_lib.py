"""Thin ctypes binding over the C ABI in include/fa.h (argument marshalling only).

Every function here maps torch tensors to device pointers and sizes and calls
the same-named entry point of ``libta11_fa.so``; all arithmetic runs in the
library's CUDA kernels.  PyTorch only provides device memory and the current
stream.  There is no fallback: if the library is missing, or the device is not
an sm_103 GB300, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libta11_fa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED_D = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_DEVICE = 5
FA_ERR_LAUNCH = 6
FA_ERR_TIMEOUT = 7
FA_ERR_SCRATCH_LIMIT = 8

EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror", "fa_device_status",
            "fa_set_wait_limit_ns", "fa_set_fwd_persistent", "fa_set_bwd_persistent", "fa_wait_probe", "fa_set_bwd_main_events", "fa_bwd_noalloc",
            "fa_graph_create", "fa_graph_launch", "fa_graph_destroy", "fa_fwd_varlen", "fa_bwd_varlen",
            "fa_bwd_varlen_workspace_size", "fa_fwd_window", "fa_bwd_window", "fa_fwd_window_workspace_size", "fa_bwd_window_workspace_size",
            "fa_quantize_e4m3",
            "fa_quantize_e4m3_transposed", "fa_quantize_qkv_e4m3", "fa_fwd_fp8", "fa_step_host",
            "fa_step_host_device_bytes")

_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


def lib() -> ctypes.CDLL:
    """Load libta11_fa.so (built in-tree by ``build.py``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.fa_fwd.restype = i
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    L.fa_bwd.restype = i
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_bwd_workspace_size.restype = sz
    L.fa_strerror.argtypes = [i]
    L.fa_strerror.restype = ctypes.c_char_p
    L.fa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
    L.fa_device_status.restype = i
    L.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    L.fa_set_wait_limit_ns.restype = None
    L.fa_set_fwd_persistent.argtypes = [i]
    L.fa_set_fwd_persistent.restype = i
    L.fa_set_bwd_persistent.argtypes = [i]
    L.fa_set_bwd_persistent.restype = i
    L.fa_wait_probe.argtypes = [ctypes.c_ulonglong, vp]
    L.fa_wait_probe.restype = i
    L.fa_set_bwd_main_events.argtypes = [vp, vp]
    L.fa_set_bwd_main_events.restype = None
    L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.fa_bwd_noalloc.restype = i
    L.fa_graph_create.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz,
                                  ctypes.POINTER(vp)]
    L.fa_graph_create.restype = i
    L.fa_graph_launch.argtypes = [vp, vp]
    L.fa_graph_launch.restype = i
    L.fa_graph_destroy.argtypes = [vp]
    L.fa_graph_destroy.restype = None
    L.fa_step_host_device_bytes.argtypes = [i, i, i, i, i]
    L.fa_step_host_device_bytes.restype = sz
    L.fa_step_host.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, i, vp]
    L.fa_step_host.restype = i
    L.fa_quantize_e4m3.argtypes = [vp, ctypes.c_longlong, vp, vp, vp, vp]
    L.fa_quantize_e4m3.restype = i
    L.fa_quantize_e4m3_transposed.argtypes = [vp, i, i, i, i, i, vp, vp, vp, vp]
    L.fa_quantize_e4m3_transposed.restype = i
    L.fa_quantize_qkv_e4m3.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp, vp, i, vp, vp, vp]
    L.fa_quantize_qkv_e4m3.restype = i
    L.fa_fwd_fp8.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.fa_fwd_fp8.restype = i
    L.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, i, vp, sz, vp]
    L.fa_fwd_window.restype = i
    L.fa_fwd_window_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    L.fa_fwd_window_workspace_size.restype = sz
    L.fa_bwd_window_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
    L.fa_bwd_window_workspace_size.restype = sz
    L.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, i, vp, sz, vp]
    L.fa_bwd_window.restype = i
    L.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    L.fa_fwd_varlen.restype = i
    L.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_bwd_varlen_workspace_size.restype = sz
    L.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
    L.fa_bwd_varlen.restype = i
    _lib = L
    return L


def strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, name: str, dtype) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"{name} is on cuda:{t.get_device()} but the library runs on the current device, "
                         f"cuda:{torch.cuda.current_device()} (select it with torch.cuda.device)")
    return t.data_ptr()


def _check(rc: int, where: str):
    if rc != FA_OK:
        raise FAError(rc, where)


# The C calls receive pointers and the sizes read from q and k, and the kernels index
# every other tensor by those sizes: a tensor of another shape would be read or written
# past its end.  So each wrapper first checks every tensor's shape against them.
def _expect(t, name: str, shape) -> None:
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dense_sizes(q, k, v, o=None, lse=None, do=None, dq=None, dk=None, dv=None):
    """(B, H, Nq, Nk, D) of [B,H,N,D] tensors, after checking that the shapes agree."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError(f"q and k must be [B, H, N, D], got {tuple(q.shape)} and {tuple(k.shape)}")
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    _expect(k, "k", (B, H, Nk, D))
    _expect(v, "v", (B, H, Nk, D))
    for t, name in ((o, "o"), (do, "do"), (dq, "dq")):
        _expect(t, name, (B, H, Nq, D))
    _expect(lse, "lse", (B, H, Nq))
    _expect(dk, "dk", (B, H, Nk, D))
    _expect(dv, "dv", (B, H, Nk, D))
    return B, H, Nq, Nk, D


def _packed_sizes(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, do=None, dq=None, dk=None, dv=None):
    """(B, H, total_q, total_k, D) of packed [total, H, D] tensors, after checking shapes."""
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError(f"q and k must be [total, H, D], got {tuple(q.shape)} and {tuple(k.shape)}")
    total_q, H, D = q.shape
    total_k = k.shape[0]
    _expect(k, "k", (total_k, H, D))
    _expect(v, "v", (total_k, H, D))
    for t, name in ((o, "o"), (do, "do"), (dq, "dq")):
        _expect(t, name, (total_q, H, D))
    _expect(lse, "lse", (H, total_q))
    _expect(dk, "dk", (total_k, H, D))
    _expect(dv, "dv", (total_k, H, D))
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() < 2:
        raise ValueError(f"cu_seqlens_q must hold B + 1 >= 2 offsets, got shape {tuple(cu_seqlens_q.shape)}")
    _expect(cu_seqlens_k, "cu_seqlens_k", tuple(cu_seqlens_q.shape))
    return cu_seqlens_q.numel() - 1, H, total_q, total_k, D


def fa_bwd_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int) -> int:
    return int(lib().fa_bwd_workspace_size(B, H, Nq, Nk, D))


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float | None = None, stream=None) -> None:
    """C ``fa_fwd`` on [B,H,N,D] bf16 tensors; writes o (bf16) and lse (fp32 [B,H,Nq])."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().fa_fwd(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16), _ptr(v, "v", torch.bfloat16),
                      _ptr(o, "o", torch.bfloat16), _ptr(lse, "lse", torch.float32),
                      B, H, Nq, Nk, D, float(scale), int(bool(causal)), _stream(stream))
    _check(rc, "fa_fwd")


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float | None = None, workspace=None,
           stream=None) -> None:
    """C ``fa_bwd``; allocates the workspace with torch when none is given."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse, do, dq, dk, dv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = fa_bwd_workspace_size(B, H, Nq, Nk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib().fa_bwd(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16), _ptr(v, "v", torch.bfloat16),
                      _ptr(o, "o", torch.bfloat16), _ptr(lse, "lse", torch.float32),
                      _ptr(do, "do", torch.bfloat16), _ptr(dq, "dq", torch.bfloat16),
                      _ptr(dk, "dk", torch.bfloat16), _ptr(dv, "dv", torch.bfloat16),
                      B, H, Nq, Nk, D, float(scale), int(bool(causal)),
                      _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(rc, "fa_bwd")


def forward(q, k, v, causal: bool, scale: float | None = None, stream=None):
    """Allocate outputs and run the forward: returns (o, lse)."""
    B, H, Nq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool, scale: float | None = None, workspace=None, stream=None):
    """Allocate gradients and run the backward: returns (dq, dk, dv)."""
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, workspace, stream)
    return dq, dk, dv


def fa_device_status(reset: bool = False):
    """(code, site) of the device status word; synchronises the device."""
    site = ctypes.c_uint(0)
    rc = lib().fa_device_status(ctypes.byref(site), int(bool(reset)))
    return rc, site.value


def fa_set_wait_limit_ns(ns: int) -> None:
    lib().fa_set_wait_limit_ns(int(ns))


def fa_set_fwd_persistent(on: bool) -> bool:
    """C ``fa_set_fwd_persistent``: the forward's schedule beyond one wave of CTAs (dense,
    packed, FP8 and window masks; persistent CTAs by default); returns the previous setting."""
    return bool(lib().fa_set_fwd_persistent(int(bool(on))))


def fa_set_bwd_persistent(on: bool) -> bool:
    """C ``fa_set_bwd_persistent``: the dense backward main kernel's schedule beyond one
    wave of CTAs (persistent CTAs by default); returns the previous setting."""
    return bool(lib().fa_set_bwd_persistent(int(bool(on))))


def fa_wait_probe(limit_ns: int, stream=None) -> None:
    _check(lib().fa_wait_probe(int(limit_ns), _stream(stream)), "fa_wait_probe")


def fa_set_bwd_main_events(begin=None, end=None) -> None:
    """Record torch.cuda.Events (already created by one .record()) around the main
    backward kernel of later fa_bwd calls; None, None turns it off."""
    b = begin.cuda_event if begin is not None else 0
    e = end.cuda_event if end is not None else 0
    lib().fa_set_bwd_main_events(b or None, e or None)


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float | None = None, stream=None) -> None:
    """C ``fa_bwd_noalloc``: the backward for callers that cannot allocate device
    memory; its scratch is a fixed 32 MiB array inside the library (see fa.h)."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse, do, dq, dk, dv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().fa_bwd_noalloc(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                              _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                              _ptr(lse, "lse", torch.float32), _ptr(do, "do", torch.bfloat16),
                              _ptr(dq, "dq", torch.bfloat16), _ptr(dk, "dk", torch.bfloat16),
                              _ptr(dv, "dv", torch.bfloat16), B, H, Nq, Nk, D, float(scale),
                              int(bool(causal)), _stream(stream))
    _check(rc, "fa_bwd_noalloc")


class StepGraph:
    """One fwd + bwd step captured as a CUDA graph (C ``fa_graph_create``) on fixed
    tensors; ``launch()`` replays it reading the tensors' current contents.  Keeps
    references to every tensor so none is freed while the graph exists."""

    def __init__(self, q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float | None = None, workspace=None):
        B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse, do, dq, dk, dv)
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if workspace is None:
            workspace = torch.empty(max(fa_bwd_workspace_size(B, H, Nq, Nk, D), 256), dtype=torch.uint8,
                                    device=q.device)
        self._keep = (q, k, v, o, lse, do, dq, dk, dv, workspace)
        h = ctypes.c_void_p(0)
        rc = lib().fa_graph_create(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                                   _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                                   _ptr(lse, "lse", torch.float32), _ptr(do, "do", torch.bfloat16),
                                   _ptr(dq, "dq", torch.bfloat16), _ptr(dk, "dk", torch.bfloat16),
                                   _ptr(dv, "dv", torch.bfloat16), B, H, Nq, Nk, D, float(scale),
                                   int(bool(causal)), _ptr(workspace, "workspace", torch.uint8),
                                   workspace.numel(), ctypes.byref(h))
        _check(rc, "fa_graph_create")
        self._h = h

    def launch(self, stream=None) -> None:
        _check(lib().fa_graph_launch(self._h, _stream(stream)), "fa_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().fa_graph_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------- varlen
def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  causal: bool, scale: float | None = None, stream=None) -> None:
    """C ``fa_fwd_varlen``: packed [total, H, D] bf16 tensors, lse [H, total_q] fp32,
    cu_seqlens int32 CUDA tensors of B + 1 offsets."""
    B, H, total_q, total_k, D = _packed_sizes(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().fa_fwd_varlen(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                             _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                             _ptr(lse, "lse", torch.float32), _ptr(cu_seqlens_q, "cu_seqlens_q", torch.int32),
                             _ptr(cu_seqlens_k, "cu_seqlens_k", torch.int32), B, H, total_q, total_k,
                             int(max_seqlen_q), int(max_seqlen_k), D, float(scale), int(bool(causal)),
                             _stream(stream))
    _check(rc, "fa_fwd_varlen")


def fa_bwd_varlen_workspace_size(B: int, H: int, total_q: int, max_seqlen_q: int, D: int) -> int:
    return int(lib().fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, D))


def fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool, scale: float | None = None, workspace=None, stream=None) -> None:
    """C ``fa_bwd_varlen``; allocates the workspace with torch when none is given."""
    B, H, total_q, total_k, D = _packed_sizes(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, do, dq, dk, dv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        workspace = torch.empty(max(fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, D), 256),
                                dtype=torch.uint8, device=q.device)
    rc = lib().fa_bwd_varlen(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                             _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                             _ptr(lse, "lse", torch.float32), _ptr(do, "do", torch.bfloat16),
                             _ptr(dq, "dq", torch.bfloat16), _ptr(dk, "dk", torch.bfloat16),
                             _ptr(dv, "dv", torch.bfloat16), _ptr(cu_seqlens_q, "cu_seqlens_q", torch.int32),
                             _ptr(cu_seqlens_k, "cu_seqlens_k", torch.int32), B, H, total_q, total_k,
                             int(max_seqlen_q), int(max_seqlen_k), D, float(scale), int(bool(causal)),
                             _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(rc, "fa_bwd_varlen")


# ----------------------------------------------------------------------------- local window + global tokens
def fa_fwd_window_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool, window_left: int,
                                 window_right: int, n_global: int) -> int:
    return int(lib().fa_fwd_window_workspace_size(B, H, Nq, Nk, D, int(bool(causal)), int(window_left),
                                                  int(window_right), int(n_global)))


def fa_fwd_window(q, k, v, o, lse, causal: bool, window_left: int, window_right: int, n_global: int,
                  scale: float | None = None, workspace=None, stream=None) -> None:
    """C ``fa_fwd_window`` on [B,H,N,D] bf16 tensors (negative window bound: unbounded);
    allocates the split workspace with torch when it is needed and none is given."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = fa_fwd_window_workspace_size(B, H, Nq, Nk, D, causal, window_left, window_right, n_global)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = 0 if workspace is None else _ptr(workspace, "workspace", torch.uint8)
    wbytes = 0 if workspace is None else workspace.numel()
    rc = lib().fa_fwd_window(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                             _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                             _ptr(lse, "lse", torch.float32), B, H, Nq, Nk, D, float(scale), int(bool(causal)),
                             int(window_left), int(window_right), int(n_global), wptr, wbytes, _stream(stream))
    _check(rc, "fa_fwd_window")


def fa_bwd_window_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int, window_left: int, window_right: int,
                                 n_global: int) -> int:
    return int(lib().fa_bwd_window_workspace_size(B, H, Nq, Nk, D, int(window_left), int(window_right),
                                                  int(n_global)))


def fa_bwd_window(q, k, v, o, lse, do, dq, dk, dv, causal: bool, window_left: int, window_right: int,
                  n_global: int, scale: float | None = None, workspace=None, stream=None) -> None:
    """C ``fa_bwd_window``; allocates the workspace with torch when none is given."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o, lse, do, dq, dk, dv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        workspace = torch.empty(max(fa_bwd_window_workspace_size(B, H, Nq, Nk, D, window_left, window_right,
                                                                 n_global), 256), dtype=torch.uint8, device=q.device)
    rc = lib().fa_bwd_window(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                             _ptr(v, "v", torch.bfloat16), _ptr(o, "o", torch.bfloat16),
                             _ptr(lse, "lse", torch.float32), _ptr(do, "do", torch.bfloat16),
                             _ptr(dq, "dq", torch.bfloat16), _ptr(dk, "dk", torch.bfloat16),
                             _ptr(dv, "dv", torch.bfloat16), B, H, Nq, Nk, D, float(scale), int(bool(causal)),
                             int(window_left), int(window_right), int(n_global),
                             _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(rc, "fa_bwd_window")


# ----------------------------------------------------------------------------- FP8 (e4m3) forward
def quantize_e4m3(x, stream=None):
    """C ``fa_quantize_e4m3`` on a bf16 CUDA tensor: returns (codes uint8, like x; amax, descale:
    one-element float32 CUDA tensors)."""
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(2, dtype=torch.float32, device=x.device)
    amax, descale = sc[0:1], sc[1:2]
    rc = lib().fa_quantize_e4m3(_ptr(x, "x", torch.bfloat16), x.numel(), _ptr(codes, "codes", torch.uint8),
                                amax.data_ptr(), descale.data_ptr(), _stream(stream))
    _check(rc, "fa_quantize_e4m3")
    return codes, amax, descale


def quantize_e4m3_transposed(v, stream=None):
    """C ``fa_quantize_e4m3_transposed`` on bf16 [B,H,N,D]: returns (codes_t uint8 [B,H,D,ldt],
    ldt, amax, descale) with ldt = N rounded up to 16."""
    B, H, N, D = v.shape
    ldt = (N + 15) // 16 * 16
    codes = torch.empty((B, H, D, ldt), dtype=torch.uint8, device=v.device)  # (every byte is written)
    sc = torch.empty(2, dtype=torch.float32, device=v.device)
    amax, descale = sc[0:1], sc[1:2]
    rc = lib().fa_quantize_e4m3_transposed(_ptr(v, "v", torch.bfloat16), B, H, N, D, ldt,
                                           _ptr(codes, "codes_t", torch.uint8), amax.data_ptr(),
                                           descale.data_ptr(), _stream(stream))
    _check(rc, "fa_quantize_e4m3_transposed")
    return codes, ldt, amax, descale


def fa_fwd_fp8(q8, k8, vt8, ldv: int, q_descale, k_descale, v_descale, o, lse, causal: bool,
               scale: float | None = None, stream=None) -> None:
    """C ``fa_fwd_fp8``: q8, k8 uint8 [B,H,N,D]; vt8 uint8 [B,H,D,ldv]; descales float32 CUDA scalars."""
    B, H, Nq, Nk, D = _dense_sizes(q8, k8, None, o, lse)
    _expect(vt8, "vt8", (B, H, D, int(ldv)))
    for t, name in ((q_descale, "q_descale"), (k_descale, "k_descale"), (v_descale, "v_descale")):
        if t.numel() < 1:
            raise ValueError(f"{name} must hold one float32")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().fa_fwd_fp8(_ptr(q8, "q8", torch.uint8), _ptr(k8, "k8", torch.uint8), _ptr(vt8, "vt8", torch.uint8),
                          int(ldv), _ptr(q_descale, "q_descale", torch.float32),
                          _ptr(k_descale, "k_descale", torch.float32), _ptr(v_descale, "v_descale", torch.float32),
                          _ptr(o, "o", torch.bfloat16), _ptr(lse, "lse", torch.float32), B, H, Nq, Nk, D,
                          float(scale), int(bool(causal)), _stream(stream))
    _check(rc, "fa_fwd_fp8")


def quantize_qkv_e4m3(q, k, v, stream=None):
    """C ``fa_quantize_qkv_e4m3`` on bf16 q [B,H,Nq,D], k, v [B,H,Nk,D]: returns (q8, k8 uint8
    like q, k; vt8 uint8 [B,H,D,ldv]; ldv = Nk rounded up to 16; amax, descale: float32 CUDA
    tensors of 3, in the order q, k, v)."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v)
    ldv = (Nk + 15) // 16 * 16
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=q.device)
    vt8 = torch.empty((B, H, D, ldv), dtype=torch.uint8, device=q.device)  # (every byte is written)
    sc = torch.empty(6, dtype=torch.float32, device=q.device)
    amax, descale = sc[0:3], sc[3:6]
    rc = lib().fa_quantize_qkv_e4m3(_ptr(q, "q", torch.bfloat16), _ptr(k, "k", torch.bfloat16),
                                    _ptr(v, "v", torch.bfloat16), B, H, Nq, Nk, D, _ptr(q8, "q8", torch.uint8),
                                    _ptr(k8, "k8", torch.uint8), _ptr(vt8, "vt8", torch.uint8), ldv,
                                    amax.data_ptr(), descale.data_ptr(), _stream(stream))
    _check(rc, "fa_quantize_qkv_e4m3")
    return q8, k8, vt8, ldv, amax, descale


def forward_fp8(q, k, v, causal: bool, scale: float | None = None, stream=None):
    """Quantise bf16 q, k, v per tensor (fa_quantize_qkv_e4m3: two kernels) and run the FP8
    forward; returns (o bf16, lse float32)."""
    q8, k8, vt8, ldv, _, sc = quantize_qkv_e4m3(q, k, v, stream)
    qd, kd, vd = sc[0:1], sc[1:2], sc[2:3]
    B, H, Nq, D = q.shape
    o = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd_fp8(q8, k8, vt8, ldv, qd, kd, vd, o, lse, causal, scale, stream)
    return o, lse


# ----------------------------------------------------------------------------- host-buffer step
def step_host_device_bytes(B: int, H: int, Nq: int, Nk: int, D: int) -> int:
    return int(lib().fa_step_host_device_bytes(B, H, Nq, Nk, D))


def _host_ptr(t: torch.Tensor, name: str, dtype) -> int:
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def step_host(q, k, v, do, o, lse, dq, dk, dv, dev_buf, causal: bool, scale: float | None = None,
              stream=None) -> None:
    """C ``fa_step_host``: host (pinned) bf16 [B,H,N,D] inputs / outputs, lse float32 [B,H,Nq];
    dev_buf a uint8 CUDA tensor of step_host_device_bytes(...) bytes."""
    B, H, Nq, Nk, D = _dense_sizes(q, k, v, o=o, lse=lse, do=do, dq=dq, dk=dk, dv=dv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    bf = torch.bfloat16
    rc = lib().fa_step_host(_host_ptr(q, "q", bf), _host_ptr(k, "k", bf), _host_ptr(v, "v", bf),
                            _host_ptr(do, "do", bf), _host_ptr(o, "o", bf), _host_ptr(lse, "lse", torch.float32),
                            _host_ptr(dq, "dq", bf), _host_ptr(dk, "dk", bf), _host_ptr(dv, "dv", bf),
                            _ptr(dev_buf, "dev_buf", torch.uint8), dev_buf.numel(), B, H, Nq, Nk, D, float(scale),
                            int(bool(causal)), _stream(stream))
    _check(rc, "fa_step_host")
