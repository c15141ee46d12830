"""CPU oracle for the linear-recurrence state update (test infrastructure).

This package is the slow, sequential, obviously-correct reference that the
GPU kernels are checked against.  It is TEST INFRASTRUCTURE: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product library (``scan_runtime_gb300``) never imports,
links or calls anything here, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, built with ``-O2
-ffp-contract=off`` so that single-precision results do not depend on the
compiler's fusion choices).  This module only builds it with ``gcc`` and
marshals numpy arrays through ``ctypes``.  ctypes releases the GIL during a
foreign call, so independent slices may be run from several Python threads.

Sources: "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
§2.1 (scan forms), §4.1-§4.3 (Mamba-2, DeltaNet, GLA), §5.1 (RWKV-7), and
"我拿同一份权重和 llama.cpp 正面比了一场：我手写的 C 内核，慢了 1.1–1.7 倍" §3.

Parity status: every routine is pinned by ``tests/test_oracle_*.py``
(closed forms, invariants, explicit matrix forms, brute force on tiny inputs,
hand-derived fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DECAY_PER_KEY = 0
DECAY_PER_HEAD = 1
DECAY_PER_KEY_GATED = 2
DECAY_PER_HEAD_GATED = 3

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (in-tree, git-ignored)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, f64, f32, p = ctypes.c_int32, ctypes.c_double, ctypes.c_float, ctypes.c_void_p
            for name in ("orc_scan_fma_f64", "orc_scan_gated_f64", "orc_scan_fma_f32", "orc_scan_gated_f32"):
                getattr(lib, name).argtypes = [i32, i32, i32, p, p, p, p, p]
                getattr(lib, name).restype = None
            lib.orc_recur_diag_f64.argtypes = [i32] * 7 + [f64] + [p] * 7
            lib.orc_recur_diag_f32.argtypes = [i32] * 7 + [f32] + [p] * 7
            lib.orc_recur_delta_f64.argtypes = [i32] * 5 + [f64] + [p] * 7
            lib.orc_recur_delta_f32.argtypes = [i32] * 5 + [f32] + [p] * 7
            lib.orc_recur_rwkv7_f64.argtypes = [i32] * 5 + [p] * 7
            lib.orc_recur_rwkv7_f32.argtypes = [i32] * 5 + [p] * 7
            for prec in ("f64", "f32"):
                getattr(lib, f"orc_scan_fma_bwd_{prec}").argtypes = [i32, i32, i32] + [p] * 8
                getattr(lib, f"orc_scan_gated_bwd_{prec}").argtypes = [i32, i32, i32] + [p] * 9
                getattr(lib, f"orc_scan_fma_bwd_{prec}").restype = None
                getattr(lib, f"orc_scan_gated_bwd_{prec}").restype = None
            i64 = ctypes.c_int64
            lib.orc_readout_norm_gate_f64.argtypes = [i64, i32, p, p, p, f64, p]
            lib.orc_readout_norm_gate_f64.restype = None
            lib.orc_readout_dskip_f64.argtypes = [i64, i32, i32, p, p, p, p]
            lib.orc_readout_dskip_f64.restype = None
            for name in ("orc_recur_diag_f64", "orc_recur_diag_f32", "orc_recur_delta_f64",
                         "orc_recur_delta_f32", "orc_recur_rwkv7_f64", "orc_recur_rwkv7_f32"):
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def _f32(x):
    x = np.asarray(x)
    if x.dtype != np.float32 or not x.flags.c_contiguous:
        raise TypeError("oracle inputs must be C-contiguous float32 arrays")
    return x


def _ptr(x):
    return None if x is None else x.ctypes.data


def _state(x, prec, shape):
    if x is None:
        return None
    dt = np.float64 if prec == "f64" else np.float32
    x = np.ascontiguousarray(np.asarray(x, dtype=dt))
    if x.shape != tuple(shape):
        raise ValueError(f"state shape {x.shape} != {tuple(shape)}")
    return x


def _scan(kind, a, b, s0, prec):
    a, b = _f32(a), _f32(b)
    if a.ndim != 3 or a.shape != b.shape:
        raise ValueError("a and b must be (B, T, N) of the same shape")
    B, T, N = a.shape
    dt = np.float64 if prec == "f64" else np.float32
    s0 = _state(s0, prec, (B, N))
    s_out = np.empty((B, T, N), dt)
    s_fin = np.empty((B, N), dt)
    fn = getattr(_load(), f"orc_scan_{kind}_{prec}")
    fn(B, T, N, _ptr(a), _ptr(b), _ptr(s0), _ptr(s_fin), _ptr(s_out))
    return s_out, s_fin


def scan_fma(a, b, s0=None, prec="f64"):
    """FMA-form scan; returns ``(s_out (B,T,N), s_final (B,N))``."""
    return _scan("fma", a, b, s0, prec)


def scan_gated(a, u, s0=None, prec="f64"):
    """Gated-form scan; returns ``(s_out (B,T,N), s_final (B,N))``."""
    return _scan("gated", a, u, s0, prec)


def _opt32(x, shape):
    if x is None:
        return None
    x = _f32(x)
    if x.shape != tuple(shape):
        raise ValueError(f"shape {x.shape} != {tuple(shape)}")
    return x


def scan_backward(kind, a, s, s0=None, gs=None, gf=None, u=None, prec="f64"):
    """Reverse (adjoint) scan: given the forward states s (B,T,N), the direct
    gradients gs = dL/ds_t (B,T,N) and gf = dL/ds_final (B,N), return
    ``(da, db_or_du, ds0)``.  ``kind`` is "fma" or "gated" (then u is needed)."""
    a = _f32(a)
    B, T, N = a.shape
    dt = np.float64 if prec == "f64" else np.float32
    s = np.ascontiguousarray(np.asarray(s, dtype=dt))
    assert s.shape == (B, T, N)
    s0 = _state(s0, prec, (B, N))
    gs = _opt32(gs, (B, T, N))
    gf = _opt32(gf, (B, N))
    da = np.empty((B, T, N), dt)
    dbu = np.empty((B, T, N), dt)
    ds0 = np.empty((B, N), dt)
    lib = _load()
    if kind == "fma":
        getattr(lib, f"orc_scan_fma_bwd_{prec}")(B, T, N, _ptr(a), _ptr(s0), _ptr(s), _ptr(gs), _ptr(gf),
                                                _ptr(da), _ptr(dbu), _ptr(ds0))
    else:
        u = _f32(u)
        getattr(lib, f"orc_scan_gated_bwd_{prec}")(B, T, N, _ptr(a), _ptr(u), _ptr(s0), _ptr(s), _ptr(gs),
                                                  _ptr(gf), _ptr(da), _ptr(dbu), _ptr(ds0))
    return da, dbu, ds0


def recur_diag(q, k, v, d, S0=None, *, H, G, decay_kind, scale, prec="f64"):
    """Diagonal-decay recurrence; q,k (B,T,G,dk), v (B,T,H,dv), d per key
    (B,T,H,dk) or per head (B,T,H); the gated kinds scale the injection by
    (1 - d).  Returns ``(o (B,T,H,dv), S (B,H,dk,dv))``."""
    q, k, v, d = _f32(q), _f32(k), _f32(v), _f32(d)
    B, T, G_, dk = k.shape
    dv = v.shape[3]
    assert G_ == G and q.shape == k.shape and v.shape == (B, T, H, dv)
    assert d.shape == ((B, T, H, dk) if decay_kind in (DECAY_PER_KEY, DECAY_PER_KEY_GATED) else (B, T, H))
    dt = np.float64 if prec == "f64" else np.float32
    S0 = _state(S0, prec, (B, H, dk, dv))
    o = np.empty((B, T, H, dv), dt)
    S = np.empty((B, H, dk, dv), dt)
    getattr(_load(), f"orc_recur_diag_{prec}")(B, T, H, G, dk, dv, decay_kind, scale,
                                                 _ptr(q), _ptr(k), _ptr(v), _ptr(d),
                                                 _ptr(S0), _ptr(S), _ptr(o))
    return o, S


def recur_delta(q, k, v, beta, S0=None, *, scale, prec="f64"):
    """DeltaNet delta rule; q,k (B,T,H,dk), v (B,T,H,dv), beta (B,T,H).
    Returns ``(o (B,T,H,dv), S (B,H,dk,dv))``."""
    q, k, v, beta = _f32(q), _f32(k), _f32(v), _f32(beta)
    B, T, H, dk = k.shape
    dv = v.shape[3]
    assert q.shape == k.shape and v.shape == (B, T, H, dv) and beta.shape == (B, T, H)
    dt = np.float64 if prec == "f64" else np.float32
    S0 = _state(S0, prec, (B, H, dk, dv))
    o = np.empty((B, T, H, dv), dt)
    S = np.empty((B, H, dk, dv), dt)
    getattr(_load(), f"orc_recur_delta_{prec}")(B, T, H, dk, dv, scale, _ptr(q), _ptr(k),
                                                  _ptr(v), _ptr(beta), _ptr(S0), _ptr(S), _ptr(o))
    return o, S


def recur_rwkv7(q, k, v, w, S0=None, *, prec="f64"):
    """RWKV-7 rank-1 removal; q,k,w (B,T,H,dk), v (B,T,H,dv).
    Returns ``(o (B,T,H,dv), S (B,H,dv,dk))``."""
    q, k, v, w = _f32(q), _f32(k), _f32(v), _f32(w)
    B, T, H, dk = k.shape
    dv = v.shape[3]
    assert q.shape == k.shape == w.shape and v.shape == (B, T, H, dv)
    dt = np.float64 if prec == "f64" else np.float32
    S0 = _state(S0, prec, (B, H, dv, dk))
    o = np.empty((B, T, H, dv), dt)
    S = np.empty((B, H, dv, dk), dt)
    getattr(_load(), f"orc_recur_rwkv7_{prec}")(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                                  _ptr(w), _ptr(S0), _ptr(S), _ptr(o))
    return o, S


def readout_norm_gate(o, g, w=None, *, eps):
    """GLA readout epilogue y = RMSNorm(o) * w * silu(g) over the last axis
    (normalised first, gated after); o, g (..., dv), w (dv,) or None.
    Returns y in float64."""
    o, g = _f32(o), _f32(g)
    assert o.shape == g.shape
    dv = o.shape[-1]
    w = None if w is None else _f32(w)
    assert w is None or w.shape == (dv,)
    y = np.empty(o.shape, np.float64)
    _load().orc_readout_norm_gate_f64(o.size // dv, dv, _ptr(o), _ptr(g), _ptr(w), float(eps), _ptr(y))
    return y


def readout_dskip(o, x, D):
    """Mamba-2 skip connection y = o + D_h x; o, x (B, T, H, dv), D (H,).
    Returns y in float64."""
    o, x, D = _f32(o), _f32(x), _f32(D)
    assert o.shape == x.shape and o.ndim == 4 and D.shape == (o.shape[2],)
    H, dv = o.shape[2], o.shape[3]
    y = np.empty(o.shape, np.float64)
    _load().orc_readout_dskip_f64(o.size // dv, H, dv, _ptr(o), _ptr(x), _ptr(D), _ptr(y))
    return y
