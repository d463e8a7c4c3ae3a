"""SwiAttn routed hybrid attention on GB300: thin Python binding of libswiattn.

Every function here marshals arguments to the C ABI declared in
``include/swiattn.h`` (same names, without the ``swiattn_`` prefix) and
returns; all computation runs in the library's CUDA kernels.  PyTorch only
provides device memory and the current stream.  There is no fallback: if the
shared library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

__all__ = [
    "SwiAttnError", "F32", "BF16", "library_path", "route", "prefill", "decode", "dual_branch",
    "prefill_workspace", "decode_workspace", "dual_branch_workspace", "get_device_error",
    "status_string", "num_sms", "set_profile_events", "EXPORTS", "prefill_backward",
    "prefill_backward_workspace", "route_backward", "route_backward_workspace", "decode_paged",
    "decode_paged_workspace", "decode_anchored", "decode_anchored_workspace",
]

F32, BF16 = 0, 1
_DT = {torch.float32: F32, torch.bfloat16: BF16}
_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libswiattn.so")
_lock = threading.Lock()
_lib = None

# Every symbol include/swiattn.h declares.
EXPORTS = (
    "swiattn_route", "swiattn_prefill_workspace", "swiattn_prefill", "swiattn_decode_workspace",
    "swiattn_decode", "swiattn_decode_noalloc", "swiattn_dual_branch_workspace",
    "swiattn_dual_branch", "swiattn_prefill_backward_workspace", "swiattn_prefill_backward",
    "swiattn_route_backward_workspace", "swiattn_route_backward",
    "swiattn_decode_paged_workspace", "swiattn_decode_paged", "swiattn_decode_anchored_workspace",
    "swiattn_decode_anchored", "swiattn_prefill_anchored", "swiattn_route_prefill_workspace",
    "swiattn_route_prefill", "swiattn_prefill_host_workspace", "swiattn_prefill_host",
    "swiattn_get_device_error", "swiattn_status_string", "swiattn_set_profile_events",
    "swiattn_num_sms", "swiattn_set_wait_limit_ns",
)


class SwiAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libswiattn.so not found at {_LIB_PATH}: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_float, ctypes.c_size_t)
            lib.swiattn_route.argtypes = [vp, vp, f32, i64, i32, i32, vp, vp, vp]
            lib.swiattn_prefill_workspace.argtypes = [i32] * 7
            lib.swiattn_prefill_workspace.restype = sz
            lib.swiattn_prefill.argtypes = [vp] * 6 + [i32] * 6 + [f32, i32, vp, sz, vp]
            lib.swiattn_decode_workspace.argtypes = [i32] * 7
            lib.swiattn_decode_workspace.restype = sz
            lib.swiattn_decode.argtypes = [vp] * 7 + [i32] * 6 + [f32, i32, vp, sz, vp]
            lib.swiattn_decode_noalloc.argtypes = [vp] * 7 + [i32] * 6 + [f32, i32, vp]
            lib.swiattn_dual_branch_workspace.argtypes = [i32] * 7
            lib.swiattn_dual_branch_workspace.restype = sz
            lib.swiattn_dual_branch.argtypes = ([vp] * 12 + [i32] * 6 + [f32] * 4
                                                + [i32, vp, sz, vp])
            lib.swiattn_prefill_backward_workspace.argtypes = [i32] * 7
            lib.swiattn_prefill_backward_workspace.restype = sz
            lib.swiattn_prefill_backward.argtypes = [vp] * 10 + [i32] * 6 + [f32, i32, vp, sz, vp]
            lib.swiattn_route_backward_workspace.argtypes = [i64, i32, i32]
            lib.swiattn_route_backward_workspace.restype = sz
            lib.swiattn_route_backward.argtypes = [vp] * 8 + [i64, i32, i32, i32] + [vp] * 5 + [sz, vp]
            lib.swiattn_decode_paged_workspace.argtypes = [i32] * 9
            lib.swiattn_decode_paged_workspace.restype = sz
            lib.swiattn_decode_paged.argtypes = [vp] * 8 + [i32] * 9 + [f32, i32, vp, sz, vp]
            lib.swiattn_decode_anchored_workspace.argtypes = [i32] * 8
            lib.swiattn_decode_anchored_workspace.restype = sz
            lib.swiattn_decode_anchored.argtypes = [vp] * 7 + [i32] * 7 + [f32, i32, vp, sz, vp]
            lib.swiattn_prefill_anchored.argtypes = [vp] * 6 + [i32] * 7 + [f32, i32, vp, sz, vp]
            lib.swiattn_prefill_host_workspace.argtypes = [i32] * 7
            lib.swiattn_prefill_host_workspace.restype = sz
            lib.swiattn_prefill_host.argtypes = [vp] * 6 + [i32] * 7 + [f32, i32, vp, sz, vp]
            lib.swiattn_route_prefill_workspace.argtypes = [i32] * 7
            lib.swiattn_route_prefill_workspace.restype = sz
            lib.swiattn_route_prefill.argtypes = ([vp, vp, f32, i32] + [vp] * 7 + [i32] * 7 +
                                                  [f32, i32, vp, sz, vp])
            lib.swiattn_get_device_error.argtypes = [vp]
            lib.swiattn_status_string.argtypes = [i32]
            lib.swiattn_status_string.restype = ctypes.c_char_p
            lib.swiattn_num_sms.argtypes = []
            lib.swiattn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.swiattn_set_profile_events.argtypes = [vp, vp]
            lib.swiattn_set_profile_events.restype = None
            for name in ("swiattn_route", "swiattn_prefill", "swiattn_decode", "swiattn_decode_noalloc",
                         "swiattn_dual_branch", "swiattn_get_device_error", "swiattn_num_sms",
                         "swiattn_prefill_backward", "swiattn_route_backward",
                         "swiattn_decode_paged", "swiattn_decode_anchored",
                         "swiattn_prefill_anchored", "swiattn_route_prefill",
                         "swiattn_prefill_host"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return _load().swiattn_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise SwiAttnError(status, where)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def num_sms() -> int:
    return int(_load().swiattn_num_sms())


def set_profile_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
    """Record start/stop around the dominant kernel of later calls (None, None: off)."""
    if start is None or stop is None:
        _load().swiattn_set_profile_events(None, None)
    else:
        _load().swiattn_set_profile_events(ctypes.c_void_p(start.cuda_event),
                                           ctypes.c_void_p(stop.cuda_event))


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the tensor-core kernels' device waits on the current device
    (0 restores the default); a failure-detection test aid."""
    _check(_load().swiattn_set_wait_limit_ns(int(ns)), "swiattn_set_wait_limit_ns")


def get_device_error() -> int:
    """Synchronise the current stream; return and clear the device error word."""
    return int(_load().swiattn_get_device_error(_stream()))


def route(h: torch.Tensor, w: torch.Tensor, bias: float, logits=None, gate=None):
    """logits = h @ w + bias (fp32), gate = logits > 0 (uint8).  h [T, D]."""
    _dev(h, "h")
    _dev(w, "w", h.dtype)
    T, D = h.shape
    logits = logits if logits is not None else torch.empty(T, device=h.device, dtype=torch.float32)
    gate = gate if gate is not None else torch.empty(T, device=h.device, dtype=torch.uint8)
    _check(_load().swiattn_route(_ptr(h), _ptr(w), float(bias), T, D, _DT[h.dtype], _ptr(logits),
                                 _ptr(gate), _stream()), "swiattn_route")
    return logits, gate


def prefill_workspace(B, N, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_prefill_workspace(B, N, Hq, Hkv, d, W, _DT.get(dtype, dtype)))


def decode_workspace(B, Lmax, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_decode_workspace(B, Lmax, Hq, Hkv, d, W, _DT.get(dtype, dtype)))


def dual_branch_workspace(B, N, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_dual_branch_workspace(B, N, Hq, Hkv, d, W, _DT.get(dtype, dtype)))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    if ws is None:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    return ws


def prefill(q, k, v, gate, W: int, scale: Optional[float] = None, out=None, want_lse=False,
            workspace=None, n_anchor: int = 0):
    """Routed prefill.  q [B,N,Hq,d], k/v [B,N,Hkv,d], gate uint8 [B,N] -> o [B,N,Hq,d].
    n_anchor > 0: window rows also see the first n_anchor keys (global anchors)."""
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    _dev(gate, "gate", torch.uint8)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, N, Hq), device=q.device, dtype=torch.float32) if want_lse else None
    nbytes = prefill_workspace(B, N, Hq, Hkv, d, W, q.dtype)
    ws = _workspace(nbytes, q.device, workspace)
    if n_anchor:
        _check(_load().swiattn_prefill_anchored(
            _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _ptr(lse), B, N, Hq, Hkv, d, W,
            n_anchor, float(scale), _DT[q.dtype], _ptr(ws), ws.numel(), _stream()),
            "swiattn_prefill_anchored")
    else:
        _check(_load().swiattn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _ptr(lse),
                                       B, N, Hq, Hkv, d, W, float(scale), _DT[q.dtype], _ptr(ws),
                                       ws.numel(), _stream()), "swiattn_prefill")
    return (o, lse) if want_lse else o


def prefill_host_workspace(B, N, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_prefill_host_workspace(B, N, Hq, Hkv, d, W, _DT.get(dtype, dtype)))


def _host(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def prefill_host(q, k, v, gate, W: int, scale: Optional[float] = None, n_anchor: int = 0,
                 out=None, want_lse=False, workspace=None, device=None):
    """Routed prefill from and to host memory (swiattn_prefill_host): q, k, v,
    gate are CPU tensors (pinned for asynchronous copies); the output is a CPU
    tensor (pinned when allocated here), valid once the current stream of
    `device` has passed the call.  workspace: a device uint8 tensor of at least
    prefill_host_workspace(...) bytes."""
    _host(q, "q")
    _host(k, "k", q.dtype)
    _host(v, "v", q.dtype)
    _host(gate, "gate", torch.uint8)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dev = torch.device(device) if device is not None else torch.device("cuda",
                                                                        torch.cuda.current_device())
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    _host(o, "out", q.dtype)
    lse = torch.empty((B, N, Hq), dtype=torch.float32, pin_memory=True) if want_lse else None
    ws = _workspace(prefill_host_workspace(B, N, Hq, Hkv, d, W, q.dtype), dev, workspace)
    with torch.cuda.device(dev):
        _check(_load().swiattn_prefill_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _ptr(lse), B, N, Hq, Hkv, d, W,
            n_anchor, float(scale), _DT[q.dtype], _ptr(ws), ws.numel(), _stream()),
            "swiattn_prefill_host")
    return (o, lse) if want_lse else o


def route_prefill_workspace(B, N, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_route_prefill_workspace(B, N, Hq, Hkv, d, W, _DT.get(dtype, dtype)))


def route_prefill(h, w, bias: float, q, k, v, W: int, scale: Optional[float] = None,
                  n_anchor: int = 0, out=None, want_lse=False, logits=None, gate=None,
                  workspace=None):
    """One layer's router and routed prefill in one call.  h [B*N, d_model] (or
    [B, N, d_model]), w [d_model]; q [B,N,Hq,d], k/v [B,N,Hkv,d].  Returns
    (o, logits fp32 [B,N], gate uint8 [B,N]) (and lse when want_lse)."""
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    _dev(h, "h", q.dtype)
    _dev(w, "w", q.dtype)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    D = h.shape[-1]
    if h.numel() != B * N * D or w.numel() != D:
        raise ValueError("h must hold B*N rows of d_model values and w d_model values")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, N, Hq), device=q.device, dtype=torch.float32) if want_lse else None
    logits = logits if logits is not None else torch.empty((B, N), device=q.device,
                                                           dtype=torch.float32)
    gate = gate if gate is not None else torch.empty((B, N), device=q.device, dtype=torch.uint8)
    ws = _workspace(route_prefill_workspace(B, N, Hq, Hkv, d, W, q.dtype), q.device, workspace)
    _check(_load().swiattn_route_prefill(
        _ptr(h), _ptr(w), float(bias), D, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(logits), _ptr(gate), B, N, Hq, Hkv, d, W, n_anchor, float(scale), _DT[q.dtype],
        _ptr(ws), ws.numel(), _stream()), "swiattn_route_prefill")
    return (o, logits, gate, lse) if want_lse else (o, logits, gate)


def decode(q, k_cache, v_cache, seq_lens, gate, W: int, scale: Optional[float] = None, out=None,
           want_lse=False, workspace=None):
    """One decode step.  q [B,Hq,d], caches [B,Lmax,Hkv,d], seq_lens int32 [B], gate uint8 [B]."""
    _dev(q, "q")
    _dev(k_cache, "k_cache", q.dtype)
    _dev(v_cache, "v_cache", q.dtype)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(gate, "gate", torch.uint8)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32) if want_lse else None
    ws = _workspace(decode_workspace(B, Lmax, Hq, Hkv, d, W, q.dtype), q.device, workspace)
    _check(_load().swiattn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                  _ptr(gate), _ptr(o), _ptr(lse), B, Lmax, Hq, Hkv, d, W,
                                  float(scale), _DT[q.dtype], _ptr(ws), ws.numel(), _stream()),
           "swiattn_decode")
    return (o, lse) if want_lse else o


def dual_branch(q, k, v, logits, nll, W: int, scale: Optional[float] = None, gamma_base=1e-3,
                eps=0.1, alpha=100.0, want_gated=True, outs=None, workspace=None, want_lse=False):
    """Dual-branch forward: dict(o_full, o_swa, o_gated, mse, gamma, reg_loss[, lse_gated])."""
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    _dev(logits, "logits", torch.float32)
    _dev(nll, "nll", torch.float32)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if outs is None:
        outs = dict(o_full=torch.empty_like(q), o_swa=torch.empty_like(q),
                    o_gated=torch.empty_like(q) if want_gated else None,
                    mse=torch.empty((B, N), device=q.device, dtype=torch.float32),
                    gamma=torch.empty((B, N), device=q.device, dtype=torch.float32),
                    reg_loss=torch.empty((B, N), device=q.device, dtype=torch.float32))
        if want_lse:
            outs["lse_gated"] = torch.empty((B, N, Hq), device=q.device, dtype=torch.float32)
    ws = _workspace(dual_branch_workspace(B, N, Hq, Hkv, d, W, q.dtype), q.device, workspace)
    _check(_load().swiattn_dual_branch(
        _ptr(q), _ptr(k), _ptr(v), _ptr(logits), _ptr(nll), _ptr(outs["o_full"]),
        _ptr(outs["o_swa"]), _ptr(outs.get("o_gated")), _ptr(outs.get("lse_gated")),
        _ptr(outs["mse"]), _ptr(outs["gamma"]),
        _ptr(outs["reg_loss"]), B, N, Hq, Hkv, d, W, float(scale), float(gamma_base), float(eps),
        float(alpha), _DT[q.dtype], _ptr(ws), ws.numel(), _stream()), "swiattn_dual_branch")
    return outs


def prefill_backward_workspace(B, N, Hq, Hkv, d, W, dtype) -> int:
    return int(_load().swiattn_prefill_backward_workspace(B, N, Hq, Hkv, d, W,
                                                          _DT.get(dtype, dtype)))


def prefill_backward(q, k, v, gate, o, lse, d_o, W: int, scale: Optional[float] = None,
                     outs=None, workspace=None):
    """Gradient of prefill: (dq, dk, dv) for output gradient d_o [B,N,Hq,d], given the
    forward's o and lse (prefill(..., want_lse=True))."""
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    _dev(gate, "gate", torch.uint8)
    _dev(o, "o", q.dtype)
    _dev(lse, "lse", torch.float32)
    _dev(d_o, "d_o", q.dtype)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = outs if outs is not None else (torch.empty_like(q), torch.empty_like(k),
                                                torch.empty_like(v))
    ws = _workspace(prefill_backward_workspace(B, N, Hq, Hkv, d, W, q.dtype), q.device, workspace)
    _check(_load().swiattn_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk),
        _ptr(dv), B, N, Hq, Hkv, d, W, float(scale), _DT[q.dtype], _ptr(ws), ws.numel(),
        _stream()), "swiattn_prefill_backward")
    return dq, dk, dv


def route_backward_workspace(tokens, d_model, dtype) -> int:
    return int(_load().swiattn_route_backward_workspace(tokens, d_model, _DT.get(dtype, dtype)))


def route_backward(logits, o_full, o_swa, d_o, gamma=None, d_reg=None, h=None, w=None,
                   want_dh=True, want_dw=True, want_db=True, workspace=None):
    """Router backward through the straight-through gate and the regulariser.
    o_full/o_swa/d_o [T, hd] (any shape with T leading rows), logits/gamma/d_reg fp32 [T],
    h [T, D], w [D].  Returns dict(d_logits[, dh, dw, db])."""
    _dev(logits, "logits", torch.float32)
    _dev(o_full, "o_full")
    _dev(o_swa, "o_swa", o_full.dtype)
    _dev(d_o, "d_o", o_full.dtype)
    T = logits.numel()
    hd = o_full.numel() // max(T, 1)
    if d_reg is not None:
        _dev(d_reg, "d_reg", torch.float32)
        _dev(gamma, "gamma", torch.float32)
    out = dict(d_logits=torch.empty(T, device=logits.device, dtype=torch.float32))
    D = 0
    if h is not None:
        _dev(h, "h", o_full.dtype)
        _dev(w, "w", o_full.dtype)
        D = w.numel()
        if want_dh:
            out["dh"] = torch.empty_like(h)
        if want_dw:
            out["dw"] = torch.empty(D, device=h.device, dtype=torch.float32)
        if want_db:
            out["db"] = torch.empty(1, device=h.device, dtype=torch.float32)
    ws = None
    if "dw" in out:
        ws = _workspace(route_backward_workspace(T, D, o_full.dtype), logits.device, workspace)
    _check(_load().swiattn_route_backward(
        _ptr(h), _ptr(w), _ptr(logits), _ptr(o_full), _ptr(o_swa), _ptr(d_o), _ptr(gamma),
        _ptr(d_reg), T, hd, D, _DT[o_full.dtype], _ptr(out["d_logits"]), _ptr(out.get("dh")),
        _ptr(out.get("dw")), _ptr(out.get("db")), _ptr(ws), 0 if ws is None else ws.numel(),
        _stream()), "swiattn_route_backward")
    return out


def decode_paged_workspace(B, max_pages, page_size, Hq, Hkv, d, W, dtype, n_anchor=0) -> int:
    return int(_load().swiattn_decode_paged_workspace(B, max_pages, page_size, Hq, Hkv, d, W,
                                                      n_anchor, _DT.get(dtype, dtype)))


def decode_anchored_workspace(B, Lmax, Hq, Hkv, d, W, n_anchor, dtype) -> int:
    return int(_load().swiattn_decode_anchored_workspace(B, Lmax, Hq, Hkv, d, W, n_anchor,
                                                         _DT.get(dtype, dtype)))


def decode_anchored(q, k_cache, v_cache, seq_lens, gate, W: int, n_anchor: int,
                    scale: Optional[float] = None, out=None, want_lse=False, workspace=None):
    """decode() where a window query also sees the first n_anchor cache entries."""
    _dev(q, "q")
    _dev(k_cache, "k_cache", q.dtype)
    _dev(v_cache, "v_cache", q.dtype)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(gate, "gate", torch.uint8)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32) if want_lse else None
    ws = _workspace(decode_anchored_workspace(B, Lmax, Hq, Hkv, d, W, n_anchor, q.dtype),
                    q.device, workspace)
    _check(_load().swiattn_decode_anchored(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(gate), _ptr(o), _ptr(lse), B,
        Lmax, Hq, Hkv, d, W, n_anchor, float(scale), _DT[q.dtype], _ptr(ws), ws.numel(),
        _stream()), "swiattn_decode_anchored")
    return (o, lse) if want_lse else o


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, gate, W: int,
                 scale: Optional[float] = None, out=None, want_lse=False, workspace=None,
                 n_anchor: int = 0):
    """Decode over a paged cache.  q [B,Hq,d]; k_pages, v_pages [num_pages, page_size, Hkv, d];
    block_table int32 [B, max_pages]; seq_lens int32 [B]; gate uint8 [B]."""
    _dev(q, "q")
    _dev(k_pages, "k_pages", q.dtype)
    _dev(v_pages, "v_pages", q.dtype)
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(gate, "gate", torch.uint8)
    B, Hq, d = q.shape
    num_pages, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_pages = block_table.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32) if want_lse else None
    ws = _workspace(decode_paged_workspace(B, max_pages, page_size, Hq, Hkv, d, W, q.dtype,
                                           n_anchor), q.device, workspace)
    _check(_load().swiattn_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(gate),
        _ptr(o), _ptr(lse), B, max_pages, page_size, num_pages, Hq, Hkv, d, W, n_anchor,
        float(scale), _DT[q.dtype], _ptr(ws), ws.numel(), _stream()), "swiattn_decode_paged")
    return (o, lse) if want_lse else o
