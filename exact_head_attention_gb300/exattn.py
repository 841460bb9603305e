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
# attn_mask: none, top-left causal (query q sees keys k <= q), bottom-right causal (k <= q + Nk - Nq)
ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 0, 1, 2
_MASKS = {False: 0, True: 1, 0: 0, 1: 1, 2: 2, "none": 0, "top_left": 1, "bottom_right": 2}
# attn_dq_mode
DQ_MODES = {"atomic": 0, "deterministic": 1, "auto": 2}
# attn_bwd is these three C-ABI calls in this order
BWD_STEPS = ("attn_bwd_preprocess", "attn_bwd_kv_blocks", "attn_bwd_dq_convert")

_lock = threading.Lock()
_lib = None


class Strides(ctypes.Structure):
    """attn_strides: element strides of a [B][H][N][d] view with contiguous d."""
    _fields_ = [("batch", ctypes.c_longlong), ("head", ctypes.c_longlong), ("row", ctypes.c_longlong)]


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
            st = Strides
            lib.attn_fwd_strided.argtypes = [vp, st, vp, st, vp, st, vp, st, vp, i, i, i, i, i, i, f, i, vp]
            lib.attn_fwd_strided.restype = i
            lib.attn_bwd_strided.argtypes = [vp, st, vp, st, vp, st, vp, st, vp, st, vp, vp, st, vp, st, vp, st,
                                             i, i, i, i, i, i, f, i, vp, sz, vp]
            lib.attn_bwd_strided.restype = i
            lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
            lib.attn_fwd_splitkv.restype = i
            lib.attn_fwd_splitkv_strided.argtypes = [vp, st, vp, st, vp, st, vp, st, vp, i, i, i, i, i, i, f, i, i, vp,
                                                     sz, vp]
            lib.attn_fwd_splitkv_strided.restype = i
            lib.attn_fwd_splitkv_num_splits.argtypes = [i, i, i, i, i, i]
            lib.attn_fwd_splitkv_num_splits.restype = i
            lib.attn_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i]
            lib.attn_fwd_splitkv_workspace_size.restype = sz
            lib.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
            lib.attn_bwd_ex.restype = i
            lib.attn_bwd_strided_ex.argtypes = [vp, st, vp, st, vp, st, vp, st, vp, st, vp, vp, st, vp, st, vp, st,
                                                i, i, i, i, i, i, f, i, i, vp, sz, vp]
            lib.attn_bwd_strided_ex.restype = i
            lib.attn_kl_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
            lib.attn_kl_fwd.restype = i
            lib.attn_kl_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, f, i, vp]
            lib.attn_kl_bwd.restype = i
            lib.attn_kl_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, f, i, i, vp,
                                           sz, vp]
            lib.attn_kl_bwd_ex.restype = i
            lib.attn_kl_bwd_workspace_size.argtypes = [i, i, i, i]
            lib.attn_kl_bwd_workspace_size.restype = sz
            lib.attn_selftest_wait_timeout.argtypes = [i, vp]
            lib.attn_selftest_wait_timeout.restype = i
            lib.attn_kl_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
            lib.attn_kl_fwd_splitkv.restype = i
            lib.attn_kl_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i]
            lib.attn_kl_fwd_splitkv_workspace_size.restype = sz
            lib.attn_fwd_schedule.argtypes = [i, i, i, i, i, i, i, vp, i, vp, i]
            lib.attn_fwd_schedule.restype = i
            lib.attn_bwd_head_group.argtypes = [i, i, i, i, i, i, i, sz]
            lib.attn_bwd_head_group.restype = i
            lib.attn_bwd_auto_dq_mode.argtypes = [i, i, i, i, i, i]
            lib.attn_bwd_auto_dq_mode.restype = i
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


def mask_code(causal) -> int:
    """attn_mask value of `causal`: False/0/"none", True/1/"top_left", 2/"bottom_right"."""
    if causal not in _MASKS:
        raise ValueError(f"unknown causal mask {causal!r}")
    return _MASKS[causal]


def _ptr(t):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _view(t):
    """(pointer, Strides) of a [B, H, N, d] CUDA tensor whose last dimension is contiguous."""
    if not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("tensors must be [B, H, N, d] CUDA tensors with a contiguous last dimension")
    return ctypes.c_void_p(t.data_ptr()), Strides(t.stride(0), t.stride(1), t.stride(2))


def _all_contiguous(*ts) -> bool:
    return all(t.is_contiguous() for t in ts)


# The current stream's raw handle without building a Stream object (several microseconds a call);
# the public call is the fallback where this accessor is absent.
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _RAW_STREAM is not None:
        return ctypes.c_void_p(_RAW_STREAM(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    return B, H, Nq, k.shape[2], d


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def fwd_raw(q, k, v, o, lse, causal, scale: float, stream=None) -> int:
    """Calls attn_fwd on caller-provided contiguous tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, mask_code(causal),
                           float(scale), _dtype_code(q), _stream(stream))


def fwd_strided_raw(q, k, v, o, lse, causal, scale: float, stream=None) -> int:
    """Calls attn_fwd_strided with each tensor's own strides; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    return load().attn_fwd_strided(*_view(q), *_view(k), *_view(v), *_view(o), _ptr(lse), B, H, Nq, Nk, d,
                                   mask_code(causal), float(scale), _dtype_code(q), _stream(stream))


def forward(q, k, v, causal=False, scale: float | None = None, stream=None):
    """O [B,H,Nq,d] (dtype and, where dense, strides of q) and LSE [B,H,Nq] fp32.

    `causal`: False, True (top-left) or "bottom_right".  Non-contiguous views whose last
    dimension is contiguous (e.g. [B, N, H, d] storage seen as [B, H, N, d]) go through
    attn_fwd_strided without a copy."""
    B, H, Nq, Nk, d = _dims(q, k)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if _all_contiguous(q, k, v, o):
        _check(fwd_raw(q, k, v, o, lse, causal, scale, stream), "attn_fwd")
    else:
        _check(fwd_strided_raw(q, k, v, o, lse, causal, scale, stream), "attn_fwd_strided")
    return o, lse


def splitkv_num_splits(B: int, H: int, Nq: int, Nk: int, d: int, sm_count: int = 0) -> int:
    """Slices per query tile attn_fwd_splitkv picks for num_splits = 0 (sm_count 0: the current device)."""
    return int(load().attn_fwd_splitkv_num_splits(B, H, Nq, Nk, d, sm_count))


def splitkv_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    return int(load().attn_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits))


def fwd_splitkv_raw(q, k, v, o, lse, causal, scale: float, num_splits: int, workspace, stream=None) -> int:
    """Calls attn_fwd_splitkv (contiguous tensors) or attn_fwd_splitkv_strided; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    common = (B, H, Nq, Nk, d, mask_code(causal), float(scale), _dtype_code(q), int(num_splits),
              *_workspace(workspace), _stream(stream))
    if _all_contiguous(q, k, v, o):
        return load().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), *common)
    return load().attn_fwd_splitkv_strided(*_view(q), *_view(k), *_view(v), *_view(o), _ptr(lse), *common)


def forward_splitkv(q, k, v, causal=False, scale: float | None = None, num_splits: int = 0, stream=None):
    """forward() for few query rows with the key dimension divided across blocks (decoding).

    num_splits = 0 lets the library choose (possibly 1, i.e. the plain forward)."""
    B, H, Nq, Nk, d = _dims(q, k)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_bytes = splitkv_workspace_size(B, H, Nq, Nk, d, num_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(fwd_splitkv_raw(q, k, v, o, lse, causal, scale, num_splits, ws, stream), "attn_fwd_splitkv")
    return o, lse


def workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return int(load().attn_bwd_workspace_size(B, H, Nq, d))


def _workspace(workspace):
    ws_ptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return ws_ptr, ws_bytes


def bwd_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale: float, workspace, stream=None,
            step: str = "attn_bwd") -> int:
    """Calls attn_bwd (or one of BWD_STEPS) on caller-provided contiguous tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    fn = getattr(load(), step)
    return fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
              B, H, Nq, Nk, d, mask_code(causal), float(scale), _dtype_code(q), *_workspace(workspace),
              _stream(stream))


def bwd_strided_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale: float, workspace, stream=None) -> int:
    """Calls attn_bwd_strided with each tensor's own strides; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    return load().attn_bwd_strided(*_view(q), *_view(k), *_view(v), *_view(o), *_view(do), _ptr(lse),
                                   *_view(dq), *_view(dk), *_view(dv), B, H, Nq, Nk, d, mask_code(causal),
                                   float(scale), _dtype_code(q), *_workspace(workspace), _stream(stream))


def fwd_schedule(B: int, H: int, Nq: int, Nk: int, d: int, causal=False, sm_count: int = 0):
    """The forward's packed lists of query blocks (attn_fwd_schedule): a list of per-CTA lists of block
    ids (bh * ceil(Nq/256) + qb), or None when the plain launch is used."""
    cap = 2048
    blocks = (ctypes.c_uint32 * cap)()
    begin = (ctypes.c_int * 256)()
    n = int(load().attn_fwd_schedule(B, H, Nq, Nk, d, mask_code(causal), sm_count, blocks, cap, begin, 256))
    if n < 0:
        raise ValueError("invalid sizes")
    if n == 0:
        return None
    return [list(blocks[begin[c]:begin[c + 1]]) for c in range(n)]


def head_group(B: int, H: int, Nq: int, Nk: int, d: int, causal=False, sm_count: int = 0, l2_bytes: int = 0) -> int:
    """Heads per launch group of the reducing backward (attn_bwd_head_group); sm_count / l2_bytes 0 take
    the current device's values."""
    g = int(load().attn_bwd_head_group(B, H, Nq, Nk, d, mask_code(causal), sm_count, l2_bytes))
    if g < 0:
        raise ValueError("invalid sizes")
    return g


def auto_dq_mode(B: int, H: int, Nq: int, Nk: int, d: int, causal=False) -> str:
    """The mode "auto" resolves to for this backward (attn_bwd_auto_dq_mode)."""
    code = int(load().attn_bwd_auto_dq_mode(B, H, Nq, Nk, d, mask_code(causal)))
    if code < 0:
        raise ValueError("invalid sizes")
    return {v: k for k, v in DQ_MODES.items()}[code]


def dq_mode_code(dq_mode) -> int:
    if isinstance(dq_mode, str):
        if dq_mode not in DQ_MODES:
            raise ValueError(f"unknown dq_mode {dq_mode!r}")
        return DQ_MODES[dq_mode]
    return int(dq_mode)


def bwd_ex_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale: float, dq_mode, workspace, stream=None) -> int:
    """Calls attn_bwd_ex (contiguous) or attn_bwd_strided_ex with a dQ mode; returns the status code."""
    B, H, Nq, Nk, d = _dims(q, k)
    common = (B, H, Nq, Nk, d, mask_code(causal), float(scale), _dtype_code(q), dq_mode_code(dq_mode),
              *_workspace(workspace), _stream(stream))
    if _all_contiguous(q, k, v, o, do, dq, dk, dv):
        return load().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), *common)
    return load().attn_bwd_strided_ex(*_view(q), *_view(k), *_view(v), *_view(o), *_view(do), _ptr(lse),
                                      *_view(dq), *_view(dk), *_view(dv), *common)


def backward(q, k, v, o, do, lse, causal=False, scale: float | None = None, workspace=None, stream=None,
             dq_mode="atomic"):
    """(dQ, dK, dV) for the loss sum(O * dO).  `workspace` (uint8 CUDA tensor) is allocated if omitted.

    dq_mode: "atomic" (attn_bwd), "deterministic" (dQ from a query-tile kernel, same bits on every
    run) or "auto".  Gradients take the strides of q, k, v where those are dense; views go through
    the strided entry points."""
    B, H, Nq, Nk, d = _dims(q, k)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(workspace_size(B, H, Nq, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if dq_mode_code(dq_mode) != DQ_MODES["atomic"]:
        _check(bwd_ex_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale, dq_mode, workspace, stream), "attn_bwd_ex")
    elif _all_contiguous(q, k, v, o, do, dq, dk, dv):
        _check(bwd_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream), "attn_bwd")
    else:
        _check(bwd_strided_raw(q, k, v, o, do, lse, dq, dk, dv, causal, scale, workspace, stream),
               "attn_bwd_strided")
    return dq, dk, dv


def selftest_wait_timeout(timeout_ms: int = 20, stream=None) -> int:
    """Runs attn_selftest_wait_timeout: a bounded device wait that nothing satisfies.  Returns the status
    (ATTN_ERR_TIMEOUT = 5 when the timeout path works)."""
    return int(load().attn_selftest_wait_timeout(int(timeout_ms), _stream(stream)))


def check_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(load().attn_check_device_error(_stream(stream)))


class _AttnFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, dq_mode):
        o, lse = forward(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.dq_mode = causal, scale, dq_mode
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        if do.stride(-1) != 1:
            do = do.contiguous()
        dq, dk, dv = backward(q, k, v, o, do, lse, ctx.causal, ctx.scale, dq_mode=ctx.dq_mode)
        return dq, dk, dv, None, None, None


def attention(q, k, v, causal=False, scale: float | None = None, dq_mode="atomic"):
    """Autograd-aware exact attention over [B, H, N, d] tensors (causal: False, True or "bottom_right";
    dq_mode: "atomic", "deterministic" or "auto")."""
    scale = (1.0 / q.shape[-1] ** 0.5) if scale is None else scale
    return _AttnFunction.apply(q, k, v, causal, scale, dq_mode)


# ------------------------------------------------------------------ attention KL divergence

KL_SETTINGS = {"student": 1, "teacher": 2, 1: 1, 2: 2}


def kl_fwd_raw(q1, k1, q2, k2, kl, lse1, lse2, causal, scale: float, stream=None) -> int:
    """Calls attn_kl_fwd on caller-provided contiguous tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    return load().attn_kl_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(kl), _ptr(lse1), _ptr(lse2), B, H, Nq,
                              Nk, d, mask_code(causal), float(scale), _dtype_code(q1), _stream(stream))


def kl_bwd_raw(q1, k1, q2, k2, kl, lse1, lse2, g, setting, dq, dk, causal, scale: float, stream=None) -> int:
    """Calls attn_kl_bwd on caller-provided contiguous tensors; returns the status code."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    return load().attn_kl_bwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(kl), _ptr(lse1), _ptr(lse2), _ptr(g),
                              KL_SETTINGS[setting], _ptr(dq), _ptr(dk), B, H, Nq, Nk, d, mask_code(causal),
                              float(scale), _dtype_code(q1), _stream(stream))


def kl_bwd_workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    """Workspace bytes of the one-pass KL backward (attn_kl_bwd_workspace_size)."""
    return int(load().attn_kl_bwd_workspace_size(B, H, Nq, d))


def kl_bwd_ex_raw(q1, k1, q2, k2, kl, lse1, lse2, g, setting, dq, dk, causal, scale: float, dq_mode, workspace,
                  stream=None) -> int:
    """Calls attn_kl_bwd_ex (dQ mode, workspace) on caller-provided contiguous tensors; returns the status."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    return load().attn_kl_bwd_ex(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(kl), _ptr(lse1), _ptr(lse2), _ptr(g),
                                 KL_SETTINGS[setting], _ptr(dq), _ptr(dk), B, H, Nq, Nk, d, mask_code(causal),
                                 float(scale), _dtype_code(q1), dq_mode_code(dq_mode), *_workspace(workspace),
                                 _stream(stream))


def kl_forward(q1, k1, q2, k2, causal=False, scale: float | None = None, stream=None):
    """Row-wise KL(P1 || P2) of the student (q2, k2) from the teacher (q1, k1): (KL, LSE1, LSE2) [B,H,Nq] fp32."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    kl, lse1, lse2 = (torch.empty((B, H, Nq), dtype=torch.float32, device=q1.device) for _ in range(3))
    _check(kl_fwd_raw(q1, k1, q2, k2, kl, lse1, lse2, causal, scale, stream), "attn_kl_fwd")
    return kl, lse1, lse2


def kl_forward_splitkv(q1, k1, q2, k2, causal=False, scale: float | None = None, num_splits: int = 0, stream=None):
    """kl_forward for few query rows with the key dimension divided across blocks (0: library's choice)."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    kl, lse1, lse2 = (torch.empty((B, H, Nq), dtype=torch.float32, device=q1.device) for _ in range(3))
    nb = int(load().attn_kl_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits))
    ws = torch.empty(nb, dtype=torch.uint8, device=q1.device) if nb else None
    st = load().attn_kl_fwd_splitkv(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(kl), _ptr(lse1), _ptr(lse2), B, H,
                                    Nq, Nk, d, mask_code(causal), float(scale), _dtype_code(q1), int(num_splits),
                                    *_workspace(ws), _stream(stream))
    _check(st, "attn_kl_fwd_splitkv")
    return kl, lse1, lse2


def kl_backward(q1, k1, q2, k2, kl, lse1, lse2, g, train="student", causal=False, scale: float | None = None,
                stream=None, dq_mode="atomic", workspace=None):
    """(dQ, dK) of sum(g * KL) for the trained distribution ("student": Q2, K2; "teacher": Q1, K1).

    dq_mode: "atomic" / "auto" (one pass over key tiles, dQ added into an fp32 accumulator; `workspace`
    is allocated if omitted) or "deterministic" (attn_kl_bwd: two launches, the same bits on every run)."""
    B, H, Nq, Nk, d = _dims(q1, k1)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    dq, dk = torch.empty_like(q1), torch.empty_like(k1)
    g = g.contiguous().float()
    if dq_mode_code(dq_mode) == DQ_MODES["deterministic"]:
        _check(kl_bwd_raw(q1, k1, q2, k2, kl, lse1, lse2, g, train, dq, dk, causal, scale, stream), "attn_kl_bwd")
        return dq, dk
    if workspace is None:
        workspace = torch.empty(kl_bwd_workspace_size(B, H, Nq, d), dtype=torch.uint8, device=q1.device)
    _check(kl_bwd_ex_raw(q1, k1, q2, k2, kl, lse1, lse2, g, train, dq, dk, causal, scale, dq_mode, workspace, stream),
           "attn_kl_bwd_ex")
    return dq, dk


class _KlFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q1, k1, q2, k2, causal, scale, train, dq_mode):
        kl, lse1, lse2 = kl_forward(q1, k1, q2, k2, causal, scale)
        ctx.save_for_backward(q1, k1, q2, k2, kl, lse1, lse2)
        ctx.causal, ctx.scale, ctx.train, ctx.dq_mode = causal, scale, train, dq_mode
        return kl

    @staticmethod
    def backward(ctx, g):
        q1, k1, q2, k2, kl, lse1, lse2 = ctx.saved_tensors
        dq, dk = kl_backward(q1, k1, q2, k2, kl, lse1, lse2, g, ctx.train, ctx.causal, ctx.scale,
                             dq_mode=ctx.dq_mode)
        if KL_SETTINGS[ctx.train] == 1:
            return None, None, dq, dk, None, None, None, None
        return dq, dk, None, None, None, None, None, None


def attention_kl(q1, k1, q2, k2, causal=False, scale: float | None = None, train="student", dq_mode="atomic"):
    """Autograd-aware row-wise KL(P1 || P2) [B,H,Nq]; gradients flow to the trained distribution only."""
    scale = (1.0 / q1.shape[-1] ** 0.5) if scale is None else scale
    return _KlFunction.apply(q1, k1, q2, k2, causal, scale, train, dq_mode)
