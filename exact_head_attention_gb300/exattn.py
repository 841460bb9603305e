"""Thin ctypes binding over libexattn.so (include/exattn.h).

Argument marshalling only: every step of attention runs in the library's
CUDA kernels.  torch supplies device memory and the current stream.  There is
no fallback: if the library is missing or fails to load, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libexattn.so")

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_MISALIGNED",
                4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT", 6: "ATTN_ERR_WORKSPACE", 7: "ATTN_ERR_NOT_IMPLEMENTED"}
ATTN_BF16, ATTN_FP16 = 0, 1
# attn_bwd is these three C-ABI calls in this order
BWD_STEPS = ("attn_bwd_preprocess", "attn_bwd_kv_blocks", "attn_bwd_dq_convert")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = last_error()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})"
                         + (f": {detail}" if detail else ""))


def last_error() -> str:
    """The library's description of its most recent failure on this thread ("" if none)."""
    return load().attn_last_error().decode()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (raises OSError if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"{path} not found: build it with exact_head_attention_gb300.build.build()")
            lib = ctypes.CDLL(path)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
            lib.attn_fwd.restype = i
            lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
            lib.attn_bwd_workspace_size.restype = sz
            for name in ("attn_bwd",) + BWD_STEPS:
                fn = getattr(lib, name)
                fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
                fn.restype = i
            lib.attn_status_string.argtypes = [i]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_check_device_error.argtypes = [vp]
            lib.attn_check_device_error.restype = i
            lib.attn_last_error.argtypes = []
            lib.attn_last_error.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16 or float16")


def _ptr(t):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    return B, H, Nq, k.shape[2], d


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def fwd_raw(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> int:
    """Calls attn_fwd on caller-provided tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, int(bool(causal)),
                           float(scale), _dtype_code(q), _stream(stream))


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """O [B,H,Nq,d] (dtype of q) and LSE [B,H,Nq] fp32."""
    B, H, Nq, Nk, d = _dims(q, k)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check(fwd_raw(q, k, v, o, lse, causal, scale, stream), "attn_fwd")
    return o, lse


def workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return int(load().attn_bwd_workspace_size(B, H, Nq, d))


def bwd_raw(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, workspace, stream=None,
            step: str = "attn_bwd") -> int:
    """Calls attn_bwd (or one of BWD_STEPS) on caller-provided tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    ws_ptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = getattr(load(), step)
    return fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
              B, H, Nq, Nk, d, int(bool(causal)), float(scale), _dtype_code(q), ws_ptr, ws_bytes, _stream(stream))


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None, workspace=None, stream=None):
    """(dQ, dK, dV) for the loss sum(O * dO).  `workspace` (uint8 CUDA tensor) is allocated if omitted."""
    B, H, Nq, Nk, d = _dims(q, k)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(workspace_size(B, H, Nq, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check(bwd_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream), "attn_bwd")
    return dq, dk, dv


def check_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(load().attn_check_device_error(_stream(stream)))


class _AttnFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = forward(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, do.contiguous(), lse, ctx.causal, ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Autograd-aware exact attention over [B, H, N, d] tensors."""
    scale = (1.0 / q.shape[-1] ** 0.5) if scale is None else scale
    return _AttnFunction.apply(q, k, v, causal, scale)
