"""fp64 CPU oracle for the SwiAttn routed-attention hot path.

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg use it; the product library never imports or links it.  It
shares no code with the CUDA path.  The arithmetic lives in ``swiattn_oracle.c``
(plain C, double precision, OpenMP over rows); this module compiles it with gcc
and wraps it for numpy arrays.

Every function takes the exact input values as float64 arrays (bf16 or fp32
inputs widen exactly) and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libswiattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP). Returns its path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        # -ffp-contract=off: no fused multiply-add, every product is rounded
        # once as written, identically on x86-64 and aarch64 hosts.
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, u8p, i64p, i32p = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p)
            lib.oracle_row_ranges.argtypes = [u8p, i64, i64, i64, i64p, i64p]
            lib.oracle_route.argtypes = [dp, dp, ctypes.c_double, i64, i64, dp, u8p]
            lib.oracle_prefill.argtypes = [dp, dp, dp, u8p] + [i64] * 6 + [ctypes.c_double, dp, dp]
            lib.oracle_prefill_rows.argtypes = ([dp, dp, dp, u8p] + [i64] * 6
                                                + [ctypes.c_double, i64p, i64, dp, dp])
            lib.oracle_decode.argtypes = ([dp, dp, dp, i32p, u8p] + [i64] * 6
                                          + [ctypes.c_double, dp, dp])
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_softplus.argtypes = [ctypes.c_double]
            lib.oracle_softplus.restype = ctypes.c_double
            lib.oracle_regulariser.argtypes = [dp, dp, dp, i64] + [ctypes.c_double] * 3 + [dp, dp]
            lib.oracle_dual.argtypes = ([dp, dp, dp, dp, dp] + [i64] * 6
                                        + [ctypes.c_double] * 4 + [dp] * 5)
            lib.oracle_dual_rows.argtypes = ([dp, dp, dp, dp, dp] + [i64] * 6
                                             + [ctypes.c_double] * 4 + [i64p, i64] + [dp] * 5)
            lib.oracle_prefill_backward.argtypes = ([dp, dp, dp, u8p, dp] + [i64] * 6
                                                    + [ctypes.c_double, dp, dp, dp])
            lib.oracle_prefill_backward_rows.argtypes = ([dp, dp, dp, u8p, dp] + [i64] * 6
                                                         + [ctypes.c_double, i64p, i64, dp])
            lib.oracle_prefill_backward_keys.argtypes = ([dp, dp, dp, u8p, dp] + [i64] * 6
                                                         + [ctypes.c_double, i64p, i64, dp, dp])
            lib.oracle_route_backward.argtypes = [dp] * 8 + [i64] * 3 + [dp] * 4
            lib.oracle_prefill_anchored.argtypes = ([dp, dp, dp, u8p] + [i64] * 7
                                                    + [ctypes.c_double, dp, dp])
            lib.oracle_decode_anchored.argtypes = ([dp, dp, dp, i32p, u8p] + [i64] * 7
                                                   + [ctypes.c_double, dp, dp])
            for name in ("oracle_row_ranges", "oracle_route", "oracle_prefill",
                         "oracle_prefill_rows", "oracle_decode", "oracle_regulariser",
                         "oracle_dual", "oracle_dual_rows", "oracle_num_threads",
                         "oracle_prefill_backward", "oracle_prefill_backward_rows",
                         "oracle_prefill_backward_keys", "oracle_route_backward",
                         "oracle_prefill_anchored", "oracle_decode_anchored"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments")


def set_num_threads(n: int) -> None:
    """Threads of the OpenMP loops that follow (timing only)."""
    _load().oracle_set_num_threads(int(n))


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_num_threads())


def row_ranges(gate, W: int):
    """Visited key range [lo, hi] of every row; gate [B,N] (0/1)."""
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, N = g.shape
    lo = np.empty((B, N), np.int64)
    hi = np.empty((B, N), np.int64)
    _check(_load().oracle_row_ranges(_ptr(g), B, N, W, _ptr(lo), _ptr(hi)), "row_ranges")
    return lo, hi


def route(h, w, bias: float):
    """Router logits and hard gates.  h [T,D], w [D] -> logits [T] f64, gate [T] u8."""
    h, w = _f64(h), _f64(w)
    T, D = h.shape
    logits = np.empty(T, np.float64)
    gate = np.empty(T, np.uint8)
    _check(_load().oracle_route(_ptr(h), _ptr(w), float(bias), T, D, _ptr(logits), _ptr(gate)),
           "route")
    return logits, gate


def prefill(q, k, v, gate, W: int, scale: float, want_lse: bool = False):
    """Routed prefill.  q [B,N,Hq,d], k/v [B,N,Hkv,d], gate [B,N] -> o [B,N,Hq,d]
    (and lse [B,N,Hq] if asked)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, N, Hq), np.float64) if want_lse else None
    _check(_load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), B, N, Hq, Hkv, d, W,
                                  float(scale), _ptr(o), _ptr(lse) if want_lse else None),
           "prefill")
    return (o, lse) if want_lse else o


def prefill_rows(q, k, v, gate, W: int, scale: float, sel, want_lse: bool = False):
    """Routed prefill on selected (b, i, h) triples -> o [nsel,d] (and lse [nsel])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 3))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    n = sel.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64) if want_lse else None
    _check(_load().oracle_prefill_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(g), B, N, Hq, Hkv, d, W,
                                       float(scale), _ptr(sel), n, _ptr(o),
                                       _ptr(lse) if want_lse else None), "prefill_rows")
    return (o, lse) if want_lse else o


def decode(q, k_cache, v_cache, seq_lens, gate, W: int, scale: float, want_lse: bool = False):
    """One query per sequence over its cache.  q [B,Hq,d], caches [B,Lmax,Hkv,d],
    seq_lens [B], gate [B] -> o [B,Hq,d] (and lse [B,Hq])."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, Hq, d = q.shape
    Lmax, Hkv = kc.shape[1], kc.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, Hq), np.float64) if want_lse else None
    _check(_load().oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(sl), _ptr(g), B, Lmax, Hq,
                                 Hkv, d, W, float(scale), _ptr(o),
                                 _ptr(lse) if want_lse else None), "decode")
    return (o, lse) if want_lse else o


def softplus(x: float) -> float:
    return float(_load().oracle_softplus(float(x)))


def regulariser(logits, nll, mse, gamma_base=1e-3, eps=0.1, alpha=100.0):
    """Adaptive weight gamma and regulariser L per token (1-D arrays)."""
    lg, nl, ms = _f64(logits).ravel(), _f64(nll).ravel(), _f64(mse).ravel()
    n = lg.size
    gamma = np.empty(n, np.float64)
    reg = np.empty(n, np.float64)
    _check(_load().oracle_regulariser(_ptr(lg), _ptr(nl), _ptr(ms), n, float(gamma_base),
                                      float(eps), float(alpha), _ptr(gamma), _ptr(reg)),
           "regulariser")
    return gamma, reg


def dual(q, k, v, logits, nll, W: int, scale: float, gamma_base=1e-3, eps=0.1, alpha=100.0):
    """Dual-branch forward.  Returns dict o_full, o_swa [B,N,Hq,d], mse, gamma, reg [B,N]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lg, nl = _f64(logits), _f64(nll)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    of, os_ = np.empty_like(q), np.empty_like(q)
    mse, gamma, reg = (np.empty((B, N), np.float64) for _ in range(3))
    _check(_load().oracle_dual(_ptr(q), _ptr(k), _ptr(v), _ptr(lg), _ptr(nl), B, N, Hq, Hkv, d,
                               W, float(scale), float(gamma_base), float(eps), float(alpha),
                               _ptr(of), _ptr(os_), _ptr(mse), _ptr(gamma), _ptr(reg)), "dual")
    return dict(o_full=of, o_swa=os_, mse=mse, gamma=gamma, reg=reg)


def dual_rows(q, k, v, logits, nll, W: int, scale: float, sel, gamma_base=1e-3, eps=0.1,
              alpha=100.0):
    """Dual branch on selected (b, i) tokens: o_full, o_swa [nsel,Hq,d], mse/gamma/reg [nsel]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lg, nl = _f64(logits), _f64(nll)
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 2))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    n = sel.shape[0]
    of = np.empty((n, Hq, d), np.float64)
    os_ = np.empty((n, Hq, d), np.float64)
    mse, gamma, reg = (np.empty(n, np.float64) for _ in range(3))
    _check(_load().oracle_dual_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(lg), _ptr(nl), B, N, Hq, Hkv,
                                    d, W, float(scale), float(gamma_base), float(eps),
                                    float(alpha), _ptr(sel), n, _ptr(of), _ptr(os_), _ptr(mse),
                                    _ptr(gamma), _ptr(reg)), "dual_rows")
    return dict(o_full=of, o_swa=os_, mse=mse, gamma=gamma, reg=reg)


def prefill_backward(q, k, v, gate, d_o, W: int, scale: float):
    """Gradient of the routed prefill for the output gradient d_o [B,N,Hq,d]:
    returns dq [B,N,Hq,d], dk, dv [B,N,Hkv,d].  Each row's gradient flows
    through the branch its (hard) gate selected."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(d_o)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    _check(_load().oracle_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(do), B, N,
                                           Hq, Hkv, d, W, float(scale), _ptr(dq), _ptr(dk),
                                           _ptr(dv)), "prefill_backward")
    return dq, dk, dv


def prefill_backward_rows(q, k, v, gate, d_o, W: int, scale: float, sel):
    """dq of selected (b, i, h) rows -> [nsel, d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(d_o)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 3))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dq = np.empty((sel.shape[0], d), np.float64)
    _check(_load().oracle_prefill_backward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(do), B,
                                                N, Hq, Hkv, d, W, float(scale), _ptr(sel),
                                                sel.shape[0], _ptr(dq)), "prefill_backward_rows")
    return dq


def prefill_backward_keys(q, k, v, gate, d_o, W: int, scale: float, sel):
    """dk, dv of selected (b, j, kv head) keys -> two [nsel, d] arrays."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(d_o)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 3))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    n = sel.shape[0]
    dk, dv = np.empty((n, d), np.float64), np.empty((n, d), np.float64)
    _check(_load().oracle_prefill_backward_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(do), B,
                                                N, Hq, Hkv, d, W, float(scale), _ptr(sel), n,
                                                _ptr(dk), _ptr(dv)), "prefill_backward_keys")
    return dk, dv


def route_backward(logits, o_full, o_swa, d_o, gamma, d_reg=None, h=None, w=None):
    """Router backward through the straight-through gate and the regulariser.
    logits/gamma/d_reg [T]; o_full/o_swa/d_o [T, HD]; h [T, D], w [D] optional.
    Returns dict d_logits [T] and, when h and w are given, dh [T, D], dw [D], db."""
    lg, of, os_, do, gm = (_f64(x) for x in (logits, o_full, o_swa, d_o, gamma))
    T = lg.size
    of, os_, do = of.reshape(T, -1), os_.reshape(T, -1), do.reshape(T, -1)
    HD = of.shape[1]
    dr = None if d_reg is None else _f64(d_reg).ravel()
    dl = np.empty(T, np.float64)
    out = dict(d_logits=dl)
    hh = ww = dh = dw = None
    db = np.zeros(1, np.float64)
    D = 0
    if h is not None:
        hh, ww = _f64(h).reshape(T, -1), _f64(w).ravel()
        D = ww.size
        dh, dw = np.empty((T, D), np.float64), np.empty(D, np.float64)
    _check(_load().oracle_route_backward(_ptr(lg), _ptr(of), _ptr(os_), _ptr(do), _ptr(gm),
                                         None if dr is None else _ptr(dr),
                                         None if hh is None else _ptr(hh),
                                         None if ww is None else _ptr(ww), T, HD, D, _ptr(dl),
                                         None if dh is None else _ptr(dh),
                                         None if dw is None else _ptr(dw),
                                         _ptr(db) if h is not None else None), "route_backward")
    if h is not None:
        out.update(dh=dh, dw=dw, db=float(db[0]))
    return out


def prefill_anchored(q, k, v, gate, W: int, S: int, scale: float, want_lse: bool = False):
    """Routed prefill where window rows also see the first S keys (global
    anchors); S = 0 is prefill()."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, N, Hq), np.float64) if want_lse else None
    _check(_load().oracle_prefill_anchored(_ptr(q), _ptr(k), _ptr(v), _ptr(g), B, N, Hq, Hkv, d,
                                           W, S, float(scale), _ptr(o),
                                           _ptr(lse) if want_lse else None), "prefill_anchored")
    return (o, lse) if want_lse else o


def decode_anchored(q, k_cache, v_cache, seq_lens, gate, W: int, S: int, scale: float,
                    want_lse: bool = False):
    """Decode where a window query also sees the first S cache entries."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    g = np.ascontiguousarray(np.asarray(gate, dtype=np.uint8))
    B, Hq, d = q.shape
    Lmax, Hkv = kc.shape[1], kc.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, Hq), np.float64) if want_lse else None
    _check(_load().oracle_decode_anchored(_ptr(q), _ptr(kc), _ptr(vc), _ptr(sl), _ptr(g), B, Lmax,
                                          Hq, Hkv, d, W, S, float(scale), _ptr(o),
                                          _ptr(lse) if want_lse else None), "decode_anchored")
    return (o, lse) if want_lse else o
