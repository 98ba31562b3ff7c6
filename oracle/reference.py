"""ctypes wrapper around the fp64 C oracle (``attn_fp64.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The C file is the definition of attention ("FlashAttention" wiki note,
section 定義: exact, not approximate), materialising each score row; the
backward is the textbook gradient of sum(O * dO).  This module only builds the
library, marshals numpy arrays and raises on an error code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_fp64.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liborattn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_fp64.c`` with gcc (-O2, OpenMP) into ``_build/liborattn.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp] + [ctypes.c_int] * 7 + [
                ctypes.c_double, ctypes.POINTER(ctypes.c_longlong)]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [dp] * 7 + [ctypes.c_int] * 7 + [ctypes.c_double]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd_off.argtypes = [dp] * 7 + [ctypes.c_int] * 7 + [ctypes.c_double, ctypes.c_longlong]
            lib.oracle_attn_bwd_off.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def attn_fwd(q, k, v, causal: bool, scale: float, qpos=None):
    """Exact attention forward in fp64.

    q: [B,H,Nq,d]; k, v: [B,Hkv,Nk,d]; returns (o [B,H,Nq,d], lse [B,H,Nq]).
    ``qpos`` (optional, int, length Nq) gives the absolute positions of the
    query rows for the causal mask, so that a subset of rows of a long
    sequence is computed exactly (rows are independent in the definition).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    assert Bk == B and dk == d and v.shape == k.shape
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    qp = None
    if qpos is not None:
        qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
        assert qpos.shape == (Nq,)
        qp = qpos.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong))
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 B, H, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), qp)
    if rc != 0:
        raise ValueError("oracle_attn_fwd failed with code %d" % rc)
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float, qoff: int = 0):
    """Analytic attention backward in fp64 for L = sum(O * dout).

    Returns (dq [B,H,Nq,d], dk [B,Hkv,Nk,d], dv [B,Hkv,Nk,d]); dk/dv of a
    grouped K/V head are summed over the query heads that share it.  For the
    causal mask, query row i sits at position i + qoff (qoff = Nk - Nq is the
    bottom-right alignment of a query block that follows earlier keys).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    assert dout.shape == q.shape and v.shape == k.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = _load().oracle_attn_bwd_off(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                     B, H, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), int(qoff))
    if rc != 0:
        raise ValueError("oracle_attn_bwd failed with code %d" % rc)
    return dq, dk, dv
