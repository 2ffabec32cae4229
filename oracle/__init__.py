"""fp64 CPU oracle for the Lightning Attention forward pass (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (``linear_attention_hybrid_fwd_b300``) never
imports it and shares no code with it.

The arithmetic lives in ``la_oracle.c`` (plain fp64 C, see its header for what each
function restates).  This module only compiles that file with gcc, loads it with
ctypes and converts arrays to contiguous float64.

What is computed (MiniMax-01 deep dive, Hugging Face blog, "Hybrid Modeling",
mechanism steps 2-4):

* ``silu``           -- step 2, ``x / (1 + e^-x)``
* ``core``           -- step 3, the causal recurrence ``S_t = S_{t-1} + k^_t^T v^_t``,
                        ``y_t = q^_t S_t`` on already-activated inputs
* ``rmsnorm_gate``   -- step 4, ``y / sqrt(mean(y^2) + eps) * sigmoid(g)`` over the
                        H*d features of a token
* ``prefill``        -- steps 2, 3, 4 in order on raw inputs
* ``decode_step``    -- the same layer for one new token against a carried state
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIB = os.path.join(_HERE, "liblaoracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``la_oracle.c`` into ``liblaoracle.so`` next to it (gcc -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.la_oracle_silu.argtypes = [_dp, _dp, ctypes.c_int64]
        lib.la_oracle_silu.restype = None
        lib.la_oracle_core.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int64, ctypes.c_int, _dp, _dp, ctypes.c_int]
        lib.la_oracle_core.restype = ctypes.c_int
        lib.la_oracle_rmsnorm_gate.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_double, _dp, _dp]
        lib.la_oracle_rmsnorm_gate.restype = None
        lib.la_oracle_prefill.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                          _dp, _dp, _dp, ctypes.c_int]
        lib.la_oracle_prefill.restype = ctypes.c_int
        lib.la_oracle_decode_step.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              _dp, _dp]
        lib.la_oracle_decode_step.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def silu(x):
    x = _f64(x)
    y = np.empty_like(x)
    _load().la_oracle_silu(_ptr(x), _ptr(y), x.size)
    return y


def core(qh, kh, vh, S0=None, want_y=True, nthreads=0):
    """Recurrence on activated inputs ``[B,N,H,d]``; returns ``(y or None, S_final)``."""
    qh, kh, vh = _f64(qh), _f64(kh), _f64(vh)
    B, N, H, d = kh.shape
    S0 = None if S0 is None else _f64(S0).reshape(B, H, d, d)
    y = np.empty((B, N, H, d)) if want_y else None
    S = np.empty((B, H, d, d))
    _load().la_oracle_core(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(S0), B, H, N, d, _ptr(y),
                           _ptr(S), nthreads)
    return y, S


def rmsnorm_gate(y, g, eps=1e-6):
    """``y, g``: ``[..., H, d]``; the norm spans the last two axes of each token."""
    y, g = _f64(y), _f64(g)
    H, d = y.shape[-2], y.shape[-1]
    rows = y.size // (H * d)
    out = np.empty_like(y)
    _load().la_oracle_rmsnorm_gate(_ptr(y), _ptr(g), rows, H * d, eps, _ptr(out), None)
    return out


def prefill(q, k, v, g, S0=None, eps=1e-6, nthreads=0):
    """Raw inputs ``[B,N,H,d]`` -> ``(out, y_prenorm, S_final)``, all fp64."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, N, H, d = q.shape
    S0 = None if S0 is None else _f64(S0).reshape(B, H, d, d)
    out = np.empty((B, N, H, d))
    y = np.empty((B, N, H, d))
    S = np.empty((B, H, d, d))
    rc = _load().la_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0), B, H, N, d,
                                   eps, _ptr(out), _ptr(y), _ptr(S), nthreads)
    if rc != 0:
        raise MemoryError("oracle prefill: allocation failed")
    return out, y, S


def decode_step(S, q, k, v, g, eps=1e-6):
    """``S [B,H,d,d]`` (not modified), ``q,k,v,g [B,H,d]`` -> ``(out, y, S_new)``."""
    S = _f64(S).copy()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, H, d = q.shape
    out = np.empty((B, H, d))
    y = np.empty((B, H, d))
    rc = _load().la_oracle_decode_step(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(g), B, H, d,
                                       eps, _ptr(out), _ptr(y))
    if rc != 0:
        raise MemoryError("oracle decode: allocation failed")
    return out, y, S
