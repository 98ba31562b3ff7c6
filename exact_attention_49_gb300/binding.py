"""Thin Python binding of the C ABI in ``include/fa.h`` (ctypes).

Argument marshalling only: every step of the attention computation runs in the
CUDA kernels of ``libfa49.so``.  PyTorch supplies device memory and streams.
There is no fallback: if the library is missing or a call fails, an exception
is raised.

The raw entry points keep the C names (``fa_fwd``, ``fa_bwd``, ...) and take
``torch.Tensor`` arguments (or ``None`` for a NULL pointer) plus the integer
sizes; ``attention_forward`` / ``attention_backward`` are conveniences that
allocate outputs and workspace with torch and check shapes and dtypes.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_MISALIGNED = -3
FA_ERR_WORKSPACE = -4
FA_ERR_CUDA = -5
FA_ERR_DEVICE_TIMEOUT = -6

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_qk": (_I, [_P] * 5 + [_I] * 7 + [_F, _P]),
    "fa_fwd_splitkv_workspace_bytes": (_S, [_I] * 7),
    "fa_fwd_splitkv": (_I, [_P] * 5 + [_I] * 7 + [_F, _I, _P, _S, _P]),
    "fa_bwd_workspace_bytes": (_S, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_qk_workspace_bytes": (_S, [_I] * 7),
    "fa_bwd_qk": (_I, [_P] * 9 + [_I] * 7 + [_F, _I, _P, _S, _P]),
    "fa_bwd": (_I, [_P] * 9 + [_I] * 6 + [_F, _I, _P, _S, _P]),
    "fa_bwd_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_main": (_I, [_P] * 7 + [_I] * 6 + [_F, _I, _P, _S, _P]),
    "fa_bwd_postprocess": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _S, _P]),
    "fa_fp8_workspace_bytes": (_S, [_I] * 5),
    "fa_fp8_workspace_layout": (_I, [_I] * 5 + [ctypes.POINTER(ctypes.c_size_t)]),
    "fa_fp8_quantize": (_I, [_P] * 4 + [_I] * 5 + [_P, _S, _P]),
    "fa_fwd_fp8": (_I, [_P, _S, _P, _P] + [_I] * 6 + [_F, _P]),
    "fa_set_option": (_I, [ctypes.c_char_p, ctypes.c_double]),
    "fa_get_option": (_I, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double)]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_device_status": (_I, [_P]),
    "fa_version": (_I, []),
    "fa_last_error_detail": (ctypes.c_char_p, []),
}


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = lib().fa_last_error_detail().decode(errors="replace")
        super().__init__("%s failed: %s (%d)%s" % (fn, status_string(status), status,
                                                   (": " + detail) if detail else ""))
        self.status = status


def library_path() -> str:
    return _build.LIB


def lib():
    """Load ``libfa49.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError("CUDA library %s is missing: build it with "
                                   "exact_attention_49_gb300.build.build()" % path)
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


# ------------------------------------------------------------------ raw C ABI
def fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, stream=None) -> int:
    return lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                        int(causal), float(scale), _stream(stream))


def fa_fwd_qk(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, stream=None) -> int:
    return lib().fa_fwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk, d,
                           int(causal), float(scale), _stream(stream))


def fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, splits) -> int:
    return int(lib().fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, int(splits)))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, splits, workspace, workspace_bytes,
                   stream=None) -> int:
    return lib().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk, d, int(causal),
                                float(scale), int(splits), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_qk_workspace_bytes(B, H, Hkv, Nq, Nk, d, deterministic) -> int:
    return int(lib().fa_bwd_qk_workspace_bytes(B, H, Hkv, Nq, Nk, d, int(deterministic)))


def fa_bwd_qk(q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale, deterministic,
              workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                           _ptr(dv), B, H, Hkv, Nq, Nk, d, int(causal), float(scale), int(deterministic),
                           _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_workspace_bytes(B, H, Hkv, N, d, deterministic) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, Hkv, N, d, int(deterministic)))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale, deterministic,
           workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                        _ptr(dv), B, H, Hkv, N, d, int(causal), float(scale), int(deterministic),
                        _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_preprocess(o, do, lse, B, H, Hkv, N, d, deterministic, workspace, workspace_bytes,
                      stream=None) -> int:
    return lib().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), B, H, Hkv, N, d, int(deterministic),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_main(q, k, v, do, lse, dk, dv, B, H, Hkv, N, d, causal, scale, deterministic,
                workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(dk), _ptr(dv),
                             B, H, Hkv, N, d, int(causal), float(scale), int(deterministic),
                             _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_postprocess(dq, B, H, Hkv, N, d, deterministic, workspace, workspace_bytes,
                       stream=None) -> int:
    return lib().fa_bwd_postprocess(_ptr(dq), B, H, Hkv, N, d, int(deterministic),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fp8_workspace_bytes(B, H, Hkv, N, d) -> int:
    return int(lib().fa_fp8_workspace_bytes(B, H, Hkv, N, d))


def fa_fp8_workspace_layout(B, H, Hkv, N, d):
    """Byte offsets (q8, k8, v8t, sq, sk, sv, vmax, total) of the FP8 workspace."""
    out = (ctypes.c_size_t * 8)()
    st = lib().fa_fp8_workspace_layout(B, H, Hkv, N, d, out)
    if st != FA_OK:
        raise FAError("fa_fp8_workspace_layout", st)
    return [int(x) for x in out]


def fa_fp8_quantize(q, k, v, signs, B, H, Hkv, N, d, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), B, H, Hkv, N, d, _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))


def fa_fwd_fp8(workspace, workspace_bytes, o, lse, B, H, Hkv, N, d, causal, scale, stream=None) -> int:
    return lib().fa_fwd_fp8(_ptr(workspace), int(workspace_bytes), _ptr(o), _ptr(lse), B, H, Hkv, N, d, int(causal),
                            float(scale), _stream(stream))


def fa_set_option(key: str, value: float) -> int:
    return lib().fa_set_option(key.encode(), float(value))


def fa_get_option(key: str) -> float:
    out = ctypes.c_double()
    st = lib().fa_get_option(key.encode(), ctypes.byref(out))
    if st != FA_OK:
        raise FAError("fa_get_option", st)
    return out.value


def fa_last_device_status(stream=None) -> int:
    return lib().fa_last_device_status(_stream(stream))


def fa_version() -> int:
    return lib().fa_version()


# ------------------------------------------------------------------ conveniences
def _check(fn, st):
    if st != FA_OK:
        raise FAError(fn, st)


def _dims(q, k):
    B, H, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("shape mismatch: q %s k %s" % (tuple(q.shape), tuple(k.shape)))
    return B, H, Hkv, Nq, Nk, d


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                      stream=None):
    """Exact attention forward on CUDA bf16 tensors q [B,H,Nq,d], k/v [B,Hkv,Nk,d].

    Returns (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq]).  With Nq != Nk a causal mask is
    aligned bottom-right (query row i sees keys 0..i + Nk - Nq)."""
    import torch
    B, H, Hkv, N, Nk, d = _dims(q, k)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA bfloat16 tensors")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if Nk == N:
        _check("fa_fwd", fa_fwd(q, k, v, out, lse, B, H, Hkv, N, d, causal, scale, stream))
    else:
        _check("fa_fwd_qk", fa_fwd_qk(q, k, v, out, lse, B, H, Hkv, N, Nk, d, causal, scale, stream))
    return out, lse


def attention_decode(q, k, v, causal: bool = False, scale: float | None = None, splits: int = 0, out=None,
                     lse=None, workspace=None, stream=None):
    """Split-KV forward (few queries against many keys), same results as attention_forward.

    q [B,H,Nq,d], k/v [B,Hkv,Nk,d] CUDA bf16; returns (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq]).
    ``splits`` = 0 lets the library choose the number of key-range splits."""
    import torch
    B, H, Hkv, N, Nk, d = _dims(q, k)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = fa_fwd_splitkv_workspace_bytes(B, H, Hkv, N, Nk, d, splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("fa_fwd_splitkv", fa_fwd_splitkv(q, k, v, out, lse, B, H, Hkv, N, Nk, d, causal, scale, splits,
                                            workspace, 0 if workspace is None else workspace.numel(), stream))
    return out, lse


def attention_backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
                       deterministic: bool = False, dq=None, dk=None, dv=None, workspace=None,
                       stream=None):
    """Exact attention backward; returns (dq, dk, dv) as bf16 tensors."""
    import torch
    B, H, Hkv, N, Nk, d = _dims(q, k)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = fa_bwd_qk_workspace_bytes(B, H, Hkv, N, Nk, d, deterministic)
    if workspace is None:
        # torch's caching allocator returns blocks aligned to at least 512 bytes
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    if Nk == N:
        _check("fa_bwd", fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                                deterministic, workspace, workspace.numel(), stream))
    else:
        _check("fa_bwd_qk", fa_bwd_qk(q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, N, Nk, d, causal, scale,
                                      deterministic, workspace, workspace.numel(), stream))
    return dq, dk, dv


def attention_forward_fp8(q, k, v, causal: bool = False, scale: float | None = None, signs=None, out=None, lse=None,
                          workspace=None, stream=None):
    """FP8 forward (d = 128): quantise q, k, v (rotating q and k by the signed Hadamard matrix
    when ``signs`` is given: a CUDA float tensor of 128 values +-1) and run attention on the
    codes.  Returns (o bf16, lse fp32, workspace)."""
    import torch
    B, H, Hkv, N, Nk, d = _dims(q, k)
    if Nk != N:
        raise ValueError("the FP8 forward takes equal query and key lengths")
    if scale is None:
        scale = d ** -0.5
    need = fa_fp8_workspace_bytes(B, H, Hkv, N, d)
    if need == 0:
        raise FAError("fa_fp8_workspace_bytes", FA_ERR_UNSUPPORTED)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("fa_fp8_quantize", fa_fp8_quantize(q, k, v, signs, B, H, Hkv, N, d, workspace, workspace.numel(), stream))
    _check("fa_fwd_fp8", fa_fwd_fp8(workspace, workspace.numel(), out, lse, B, H, Hkv, N, d, causal, scale, stream))
    return out, lse, workspace
