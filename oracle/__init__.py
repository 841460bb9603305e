"""Exact attention oracle -- TEST INFRASTRUCTURE ONLY.

Plain single-threaded fp64 CPU attention (forward and backward) compiled from
``attn_oracle.c`` with gcc and called through ctypes.  Only the tests, the
smoke check and the benchmark's CPU-baseline leg import this package; the
product path (the CUDA library and its binding) never does, and the two share
no code.

Definitions (cited in ``attn_oracle.c``):
  * forward  O = softmax(scale * Q K^T [+ causal mask]) V
    -- SparkAttention (arXiv 2502.12784), Equation 1; CANN ops-transformer MHA
    article, section 1;
  * causal = 1 (or True, "top_left"): query q sees keys k <= q;
    causal = 2 ("bottom_right"): the queries are the last Nq positions of the
    Nk-long sequence (SparkAttention Figure 1, masked self-attention over
    preceding positions), so query q sees keys k <= q + Nk - Nq; a row that
    sees no key has O = 0, LSE = -inf and zero gradients;
  * LSE_q = m_q + ln sum_k exp(s_qk - m_q) -- StreamKL summary, Methodology 1-2;
  * backward of sum(O * dO): dV = P^T dO, dP = dO V^T, D = rowsum(P o dP),
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q -- SparkAttention,
    Figure 9 / Equation 4 (equation body not printed; exact gradient written out).

Attention KL divergence (StreamKL summary, Methodology 1-2): a teacher (1) and a
student (2) distribution P_t = softmax(scale Q_t K_t^T), KL_q = sum_k P1 (log P1 -
log P2) with log P_t = S_t - LSE_t, and the gradients of sum_q g_q KL_q for the
student (setting 1: dS2 = g (P2 - P1)) or the teacher (setting 2: dS1 = g P1
(log P1 - log P2 - KL)), dQ_t = scale dS_t K_t, dK_t = scale dS_t^T Q_t.

Every function here is pinned by tests that do not re-type the formula:
closed forms, invariants, finite differences and a library special case
(torch's fp64 CPU scaled_dot_product_attention).

Arrays are numpy float64, C-contiguous, layout [B, H, N, d]; LSE/D are [B, H, Nq].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (plain -O2, no fast-math, no threads)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            I, L, D = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, I, I, L, L, I, I, D]
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, I, I, L, L, I, I, D]
            lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, I, I, L, L, I, I, D, L, lp, dp, dp]
            lib.oracle_attn_dq_rows.argtypes = [dp, dp, dp, dp, I, I, L, L, I, I, D, L, lp, dp, dp]
            lib.oracle_attn_dkdv_cols.argtypes = [dp, dp, dp, dp, I, I, L, L, I, I, D, L, lp, dp, dp]
            lib.oracle_attn_dkdv_cols_part.argtypes = [dp, dp, dp, dp, I, I, L, L, I, I, D, L, lp, L, L, dp, dp]
            lib.oracle_attn_probs.argtypes = [dp, dp, L, L, I, I, D, dp, dp]
            lib.oracle_kl_fwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, I, I, L, L, I, I, D]
            lib.oracle_kl_bwd.argtypes = [dp, dp, dp, dp, dp, I, dp, dp, I, I, L, L, I, I, D]
            lib.oracle_kl_fwd_rows.argtypes = [dp, dp, dp, dp, I, I, L, L, I, I, D, L, lp, dp, dp, dp]
            lib.oracle_kl_dq_rows.argtypes = [dp, dp, dp, dp, dp, I, I, I, L, L, I, I, D, L, lp, dp]
            lib.oracle_kl_dk_cols.argtypes = [dp, dp, dp, dp, dp, I, I, I, L, L, I, I, D, L, lp, dp]
            lib.oracle_kl_dk_cols_part.argtypes = [dp, dp, dp, dp, dp, I, I, I, L, L, I, I, D, L, lp, L, L, dp]
            for f in (lib.oracle_attn_fwd, lib.oracle_attn_bwd, lib.oracle_attn_fwd_rows,
                      lib.oracle_attn_dq_rows, lib.oracle_attn_dkdv_cols, lib.oracle_attn_dkdv_cols_part,
                      lib.oracle_attn_probs,
                      lib.oracle_kl_fwd, lib.oracle_kl_bwd, lib.oracle_kl_fwd_rows, lib.oracle_kl_dq_rows,
                      lib.oracle_kl_dk_cols, lib.oracle_kl_dk_cols_part):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (bf16/fp16/fp32 -> fp64 is exact)."""
    if hasattr(x, "detach"):  # a torch tensor: go through fp32, which holds bf16/fp16 exactly
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _lptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


_MASKS = {False: 0, True: 1, 0: 0, 1: 1, 2: 2, "none": 0, "top_left": 1, "bottom_right": 2}


def _mask(causal) -> int:
    """Mask code: 0 none, 1 top-left causal, 2 bottom-right causal."""
    key = causal.item() if isinstance(causal, np.generic) else causal
    if key not in _MASKS:
        raise ValueError(f"unknown causal mask {causal!r}")
    return _MASKS[key]


def _shape(q, k):
    B, H, Nq, d = q.shape
    Bk, Hk, Nk, dk = k.shape
    if (B, H, d) != (Bk, Hk, dk):
        raise ValueError("q and k disagree in B, H or d")
    return B, H, Nq, Nk, d


def attn_fwd(q, k, v, causal, scale: float):
    """O [B,H,Nq,d] and LSE [B,H,Nq] in fp64 for the full problem."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, Nk, d = _shape(q, k)
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 B, H, Nq, Nk, d, _mask(causal), float(scale))
    if rc != 0:
        raise MemoryError("oracle_attn_fwd failed")
    return o, lse


def attn_bwd(q, k, v, do, causal, scale: float):
    """(dQ, dK, dV, D) in fp64 for the loss sum(O * dO)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, Nk, d = _shape(q, k)
    dq = np.zeros((B, H, Nq, d))
    dk = np.zeros((B, H, Nk, d))
    dv = np.zeros((B, H, Nk, d))
    D = np.zeros((B, H, Nq))
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(D), B, H, Nq, Nk, d, _mask(causal), float(scale))
    if rc != 0:
        raise MemoryError("oracle_attn_bwd failed")
    return dq, dk, dv, D


def attn_fwd_rows(q, k, v, causal, scale: float, rows):
    """O and LSE for chosen query rows; rows[i] = (b*H + h)*Nq + q."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, Nk, d = _shape(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    rc = _load().oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Nq, Nk, d, _mask(causal),
                                      float(scale), len(rows), _lptr(rows), _ptr(o), _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle_attn_fwd_rows failed")
    return o, lse


def attn_dq_rows(q, k, v, do, causal, scale: float, rows):
    """dQ and D for chosen query rows; rows[i] = (b*H + h)*Nq + q."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, Nk, d = _shape(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((len(rows), d))
    D = np.zeros(len(rows))
    rc = _load().oracle_attn_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, Nq, Nk, d,
                                     _mask(causal), float(scale), len(rows), _lptr(rows), _ptr(dq), _ptr(D))
    if rc != 0:
        raise MemoryError("oracle_attn_dq_rows failed")
    return dq, D


def attn_dkdv_cols(q, k, v, do, causal, scale: float, cols, q_range=None):
    """dK and dV for chosen key rows; cols[i] = (b*H + h)*Nk + k.

    q_range = (q_lo, q_hi) keeps only the contributions of query rows q_lo <= q < q_hi (dK and dV are sums
    over query rows; the parts of a partition of the rows add up to the whole)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, Nk, d = _shape(q, k)
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dk = np.zeros((len(cols), d))
    dv = np.zeros((len(cols), d))
    lo, hi = (0, Nq) if q_range is None else (int(q_range[0]), int(q_range[1]))
    rc = _load().oracle_attn_dkdv_cols_part(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, Nq, Nk, d,
                                            _mask(causal), float(scale), len(cols), _lptr(cols), lo, hi,
                                            _ptr(dk), _ptr(dv))
    if rc != 0:
        raise MemoryError("oracle_attn_dkdv_cols_part failed")
    return dk, dv


def attn_probs(qh, kh, causal, scale: float):
    """P [Nq, Nk] and LSE [Nq] of one head (qh [Nq, d], kh [Nk, d])."""
    qh, kh = _f64(qh), _f64(kh)
    Nq, d = qh.shape
    Nk = kh.shape[0]
    p = np.zeros((Nq, Nk))
    lse = np.zeros(Nq)
    _load().oracle_attn_probs(_ptr(qh), _ptr(kh), Nq, Nk, d, _mask(causal), float(scale), _ptr(p), _ptr(lse))
    return p, lse


# ---------------------------------------------------------------- attention KL divergence

def _kl_shape(q1, k1, q2, k2):
    B, H, Nq, Nk, d = _shape(q1, k1)
    if q2.shape != q1.shape or k2.shape != k1.shape:
        raise ValueError("teacher and student tensors disagree in shape")
    return B, H, Nq, Nk, d


def _setting(setting) -> int:
    if setting not in (1, 2):
        raise ValueError("setting must be 1 (student trained) or 2 (teacher trained)")
    return int(setting)


def kl_fwd(q1, k1, q2, k2, causal, scale: float):
    """KL [B,H,Nq] of the student (q2, k2) from the teacher (q1, k1), and LSE1, LSE2 [B,H,Nq]."""
    q1, k1, q2, k2 = _f64(q1), _f64(k1), _f64(q2), _f64(k2)
    B, H, Nq, Nk, d = _kl_shape(q1, k1, q2, k2)
    kl, lse1, lse2 = (np.zeros((B, H, Nq)) for _ in range(3))
    rc = _load().oracle_kl_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(kl), _ptr(lse1), _ptr(lse2),
                               B, H, Nq, Nk, d, _mask(causal), float(scale))
    if rc != 0:
        raise MemoryError("oracle_kl_fwd failed")
    return kl, lse1, lse2


def kl_bwd(q1, k1, q2, k2, g, setting, causal, scale: float):
    """(dQ, dK) of sum_q g_q KL_q for the student (setting 1) or the teacher (setting 2)."""
    q1, k1, q2, k2, g = _f64(q1), _f64(k1), _f64(q2), _f64(k2), _f64(g)
    B, H, Nq, Nk, d = _kl_shape(q1, k1, q2, k2)
    dq, dk = np.zeros((B, H, Nq, d)), np.zeros((B, H, Nk, d))
    rc = _load().oracle_kl_bwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(g), _setting(setting), _ptr(dq),
                               _ptr(dk), B, H, Nq, Nk, d, _mask(causal), float(scale))
    if rc != 0:
        raise MemoryError("oracle_kl_bwd failed")
    return dq, dk


def kl_fwd_rows(q1, k1, q2, k2, causal, scale: float, rows):
    """KL, LSE1, LSE2 of chosen rows; rows[i] = (b*H + h)*Nq + q."""
    q1, k1, q2, k2 = _f64(q1), _f64(k1), _f64(q2), _f64(k2)
    B, H, Nq, Nk, d = _kl_shape(q1, k1, q2, k2)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    kl, lse1, lse2 = (np.zeros(len(rows)) for _ in range(3))
    rc = _load().oracle_kl_fwd_rows(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), B, H, Nq, Nk, d, _mask(causal),
                                    float(scale), len(rows), _lptr(rows), _ptr(kl), _ptr(lse1), _ptr(lse2))
    if rc != 0:
        raise MemoryError("oracle_kl_fwd_rows failed")
    return kl, lse1, lse2


def kl_dq_rows(q1, k1, q2, k2, g, setting, causal, scale: float, rows):
    """dQ of the trained distribution for chosen rows; rows[i] = (b*H + h)*Nq + q."""
    q1, k1, q2, k2, g = _f64(q1), _f64(k1), _f64(q2), _f64(k2), _f64(g)
    B, H, Nq, Nk, d = _kl_shape(q1, k1, q2, k2)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((len(rows), d))
    rc = _load().oracle_kl_dq_rows(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(g), _setting(setting), B, H, Nq,
                                   Nk, d, _mask(causal), float(scale), len(rows), _lptr(rows), _ptr(dq))
    if rc != 0:
        raise MemoryError("oracle_kl_dq_rows failed")
    return dq


def kl_dk_cols(q1, k1, q2, k2, g, setting, causal, scale: float, cols, q_range=None):
    """dK of the trained distribution for chosen key rows; cols[i] = (b*H + h)*Nk + k.

    q_range = (q_lo, q_hi) keeps only the contributions of query rows q_lo <= q < q_hi."""
    q1, k1, q2, k2, g = _f64(q1), _f64(k1), _f64(q2), _f64(k2), _f64(g)
    B, H, Nq, Nk, d = _kl_shape(q1, k1, q2, k2)
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dk = np.zeros((len(cols), d))
    lo, hi = (0, Nq) if q_range is None else (int(q_range[0]), int(q_range[1]))
    rc = _load().oracle_kl_dk_cols_part(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(g), _setting(setting), B, H,
                                        Nq, Nk, d, _mask(causal), float(scale), len(cols), _lptr(cols), lo, hi,
                                        _ptr(dk))
    if rc != 0:
        raise MemoryError("oracle_kl_dk_cols_part failed")
    return dk
