"""ctypes wrapper around ``attn_oracle.c`` (test infrastructure only).

The C file is the oracle: a plain float64 evaluation of exact attention,
    O = softmax(scale * Q K^T [causal: key j <= query i]) V,  LSE = m + log l,
as defined by the forward kernel of "flash_attention_2.cu"
(leloykun/flash-hyperbolic-attention-minimal).  This module only compiles it
with the host C compiler and marshals numpy arrays; it holds none of the
method's arithmetic.

Inputs are float32 arrays holding the exact values the GPU reads (bf16 inputs
widened without rounding).  Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()


def lib_path(build_dir: str | None = None) -> str:
    return os.path.join(build_dir or _BUILD_DIR, "liboracle.so")


def build(src: str | None = None, build_dir: str | None = None, force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    src = src or _SRC
    out = lib_path(build_dir)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)
_LONGP = ctypes.POINTER(ctypes.c_long)
_L = ctypes.c_long


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _LIB
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _LIB = lib
    return _LIB


def _declare(lib):
    lib.oracle_attn_fwd.argtypes = [_F32P, _F32P, _F32P, _F64P, _F64P,
                                    _L, _L, _L, _L, _L, ctypes.c_double,
                                    ctypes.c_int, ctypes.c_int]
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [_F32P, _F32P, _F32P, _LONGP, _L, _F64P, _F64P,
                                     _L, _L, _L, _L, _L, ctypes.c_double,
                                     ctypes.c_int, ctypes.c_int]
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_probs.argtypes = [_F32P, _F32P, _F64P, _L, _L, _L, _L, _L,
                                      ctypes.c_double, ctypes.c_int]
    lib.oracle_attn_probs.restype = ctypes.c_int
    lib.oracle_attn_fwd_online.argtypes = [_F32P, _F32P, _F32P, _F64P, _F64P,
                                           _L, _L, _L, _L, _L, ctypes.c_double,
                                           ctypes.c_int, _L]
    lib.oracle_attn_fwd_online.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [_F32P, _F32P, _F32P, _F32P, _F64P, _F64P, _F64P,
                                    _L, _L, _L, _L, _L, ctypes.c_double, ctypes.c_int,
                                    ctypes.c_int]
    lib.oracle_attn_bwd.restype = ctypes.c_int


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if a.ndim != 4:
        raise ValueError("expected a [B, H, N, d] array")
    return a


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _shapes(q, k, v):
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("q [B,H,Nq,d], k and v [B,H,Nk,d] expected")
    return B, H, Nq, k.shape[2], d


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def attn_fwd(q, k, v, scale: float, causal: bool, nthreads: int | None = None,
             lib=None):
    """Full forward: returns (O [B,H,Nq,d] float64, LSE [B,H,Nq] float64)."""
    lib = lib or load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, Nq, Nk, d = _shapes(q, k, v)
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = lib.oracle_attn_fwd(_ptr(q, _F32P), _ptr(k, _F32P), _ptr(v, _F32P),
                             _ptr(o, _F64P), _ptr(lse, _F64P),
                             B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                             _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed")
    return o, lse


def attn_rows(q, k, v, rows, scale: float, causal: bool,
              nthreads: int | None = None, lib=None):
    """Selected rows (flat ids (b*H+h)*Nq+i): returns (O [n,d], LSE [n])."""
    lib = lib or load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, Nq, Nk, d = _shapes(q, k, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.dtype("long"))
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = lib.oracle_attn_rows(_ptr(q, _F32P), _ptr(k, _F32P), _ptr(v, _F32P),
                              _ptr(rows, _LONGP), n, _ptr(o, _F64P), _ptr(lse, _F64P),
                              B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                              _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_rows failed")
    return o, lse


def attn_probs(q, k, scale: float, causal: bool, lib=None):
    """Probability matrix P [B,H,Nq,Nk] (tiny problems only)."""
    lib = lib or load()
    q, k = _f32(q), _f32(k)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    p = np.empty((B, H, Nq, Nk), np.float64)
    rc = lib.oracle_attn_probs(_ptr(q, _F32P), _ptr(k, _F32P), _ptr(p, _F64P),
                               B, H, Nq, Nk, d, float(scale), int(bool(causal)))
    if rc != 0:
        raise RuntimeError("oracle_attn_probs failed")
    return p


def attn_fwd_online(q, k, v, scale: float, causal: bool, bc: int = 128, lib=None):
    """Online-softmax recurrence over bc-key tiles (for pinning only)."""
    lib = lib or load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, Nq, Nk, d = _shapes(q, k, v)
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = lib.oracle_attn_fwd_online(_ptr(q, _F32P), _ptr(k, _F32P), _ptr(v, _F32P),
                                    _ptr(o, _F64P), _ptr(lse, _F64P),
                                    B, H, Nq, Nk, d, float(scale),
                                    int(bool(causal)), int(bc))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd_online failed")
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, causal: bool, nthreads: int | None = None, lib=None):
    """Gradients (dQ, dK, dV), float64, for upstream gradient dout [B,H,Nq,d]."""
    lib = lib or load()
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, Nq, Nk, d = _shapes(q, k, v)
    if dout.shape != q.shape:
        raise ValueError("dout must have the shape of q")
    dq = np.empty(q.shape, np.float64)
    dk = np.empty(k.shape, np.float64)
    dv = np.empty(v.shape, np.float64)
    rc = lib.oracle_attn_bwd(_ptr(q, _F32P), _ptr(k, _F32P), _ptr(v, _F32P), _ptr(dout, _F32P),
                             _ptr(dq, _F64P), _ptr(dk, _F64P), _ptr(dv, _F64P),
                             B, H, Nq, Nk, d, float(scale), int(bool(causal)), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd failed")
    return dq, dk, dv
