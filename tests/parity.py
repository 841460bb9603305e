"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 CPU oracle on the same seeded inputs.

Tolerances (fixed by the method's numeric contract):
  forward O  max-abs  <= 1e-2 (bf16) / 2e-3 (fp16), for the value before its
             final rounding to the 16-bit output: |O - O_ref| may exceed the
             bound by at most half a unit in the last place of the output
             format at |O| (the correctly rounded exact result itself is that
             far away: 1.6e-2 for bf16 at |O| >= 4, where the stated bound
             alone could not be met by any 16-bit output)
  LSE        max-abs  <= 1e-3
  dQ, dK, dV relative L2 <= 2e-2
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

O_TOL = {"bf16": 1e-2, "fp16": 2e-3}
LSE_TOL = 1e-3
GRAD_TOL = 2e-2


def run_gpu(w: workloads.Workload, x: dict, backward: bool = True):
    """Forward (+ backward) on cuda through the C ABI; results copied back to CPU fp32."""
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = exattn.forward(q, k, v, w.causal, w.scale)
    out = {"o": o, "lse": lse}
    if backward:
        do = x["do"].to(dev)
        dq, dk, dv = exattn.backward(q, k, v, o, do, lse, w.causal, w.scale)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    status = exattn.check_device_error()
    assert status == 0, f"device error word: {exattn.STATUS_NAMES.get(status)}"
    return {key: t.float().cpu().numpy() for key, t in out.items()}


def rel_l2(a, b) -> float:
    """||a - b|| / ||b||, with ||b|| floored at 1e-3 * sqrt(numel): where the exact gradient is 0
    (one visible key gives dQ = dK = 0) this bounds the RMS error by 2e-5 instead of dividing by 0."""
    b = np.asarray(b, np.float64)
    floor = 1e-3 * np.sqrt(max(b.size, 1))
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), floor))


def half_ulp(x, dtype: str) -> np.ndarray:
    """Half a unit in the last place of the 16-bit format (bf16: 8 significant bits, fp16: 11) at |x|:
    the largest error of rounding to nearest there (subnormal spacing below the smallest normal)."""
    mant, emin = (7, -126) if dtype == "bf16" else (10, -14)
    e = np.floor(np.log2(np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** emin)))
    return 0.5 * 2.0 ** (e - mant)


def check_fwd(w, got_o, got_lse, ref_o, ref_lse, what=""):
    # Rows that see no key (bottom-right mask, Nq > Nk): exactly O = 0 and LSE = -inf.
    empty = np.isneginf(ref_lse)
    if empty.any():
        assert np.isneginf(got_lse[empty]).all(), f"{what}: LSE of rows without keys is not -inf"
        assert (got_o[empty] == 0).all(), f"{what}: O of rows without keys is not 0"
        got_o, got_lse, ref_o, ref_lse = got_o[~empty], got_lse[~empty], ref_o[~empty], ref_lse[~empty]
    assert np.isfinite(got_o).all() and np.isfinite(got_lse).all(), f"{what}: non-finite output"
    diff = np.abs(got_o.astype(np.float64) - ref_o)
    err_o = float(diff.max()) if ref_o.size else 0.0
    err_l = float(np.abs(got_lse - ref_lse).max()) if ref_lse.size else 0.0
    # The bound applies to the value before its final rounding to the output dtype: allow half an ulp of the
    # output format on top (taken at the larger of |O| and |O_ref|, so a value rounded across a binade
    # boundary is measured in the wider spacing).
    slack = half_ulp(np.maximum(np.abs(got_o), np.abs(ref_o)), w.dtype)
    over = diff - (O_TOL[w.dtype] + slack)
    if ref_o.size and over.max() > 0:
        i = np.unravel_index(int(np.argmax(over)), diff.shape)
        raise AssertionError(f"{what}: O error {diff[i]:.3e} at {i} (|O_ref| = {abs(ref_o[i]):.4f}) exceeds "
                             f"{O_TOL[w.dtype]} + half an ulp ({slack[i]:.2e}); plain max-abs {err_o:.3e}, "
                             f"{int((diff > O_TOL[w.dtype]).sum())} elements above {O_TOL[w.dtype]}")
    assert err_l <= LSE_TOL, f"{what}: LSE max-abs {err_l:.3e} > {LSE_TOL}"
    return err_o, err_l


def check_grads(got: dict, ref: dict, what=""):
    errs = {}
    for name in ("dq", "dk", "dv"):
        if name not in ref:
            continue
        assert np.isfinite(got[name]).all(), f"{what}: non-finite {name}"
        errs[name] = rel_l2(got[name], ref[name])
        assert errs[name] <= GRAD_TOL, f"{what}: {name} rel-L2 {errs[name]:.3e} > {GRAD_TOL}"
    return errs


def oracle_heads(w, x, heads, backward=True):
    """Full oracle on a subset of (b, h) heads; returns arrays [len(heads), N, d]."""
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])[None]  # noqa: E731  -> [1, nh, N, d]
    q, k, v = sel(x["q"]), sel(x["k"]), sel(x["v"])
    o, lse = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    ref = {"o": o[0], "lse": lse[0]}
    if backward:
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, sel(x["do"]), w.causal, w.scale)
        ref.update(dq=dq[0], dk=dk[0], dv=dv[0])
    return ref


def pick_heads(w, n=2):
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    if len(all_heads) <= n:
        return all_heads
    return [all_heads[0], all_heads[-1]][:n]


def sample_rows(N: int, n: int, seed: int) -> np.ndarray:
    """First, last and random rows in between (sorted, unique)."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 127, 128, N // 2, N - 2, N - 1]
    rows = set(r for r in fixed if 0 <= r < N)
    rows.update(rng.integers(0, N, size=max(0, n - len(rows))).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def heavy_cols(Nk: int) -> np.ndarray:
    """Key rows of the first key blocks and one in the middle.  Under a causal mask the first keys are seen by
    every query row, so their dK/dV sum over all query tiles: the longest accumulations in the backward."""
    return np.array(sorted({c for c in (0, 1, 127, 128, Nk // 2) if 0 <= c < Nk}), dtype=np.int64)


def query_parts(Nq: int, Nk: int, causal, parts: int):
    """Split the query rows [0, Nq) into `parts` ranges of about equal oracle work (a row costs its visible
    keys)."""
    q = np.arange(Nq, dtype=np.int64)
    off = Nk - Nq if causal == "bottom_right" else 0
    cost = np.clip(q + off + 1, 0, Nk) if causal else np.full(Nq, Nk)
    cum = np.cumsum(cost + 1)
    cuts = np.searchsorted(cum, cum[-1] * np.arange(1, parts) / parts).tolist()
    edges = sorted({0, Nq, *[min(max(c, 0), Nq) for c in cuts]})
    return list(zip(edges[:-1], edges[1:]))


def oracle_cols_threaded(fn, Nq: int, Nk: int, causal, workers: int | None = None):
    """Sum fn(q_range) over a partition of the query rows, the parts on a thread pool.

    fn is a column-sampled oracle call (dK/dV of chosen key rows restricted to query rows in q_range); the
    oracle's C code runs without holding the GIL, so the parts run on separate cores.  The parts of a
    partition add up to the whole sum over query rows (pinned on CPU)."""
    workers = workers or max(1, min(16, len(os.sched_getaffinity(0))))
    parts = query_parts(Nq, Nk, causal, workers)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(fn, parts))
    if isinstance(results[0], tuple):
        return tuple(sum(r[i] for r in results) for i in range(len(results[0])))
    return sum(results)


def f64_head(t, b: int, h: int) -> np.ndarray:
    """One head of a [B, H, N, d] (or [B, H, N]) tensor as a contiguous fp64 array with B = H = 1 (exact)."""
    return np.ascontiguousarray(t[b:b + 1, h:h + 1].double().cpu().numpy())


def _workers(workers=None) -> int:
    return workers or max(1, min(16, len(os.sched_getaffinity(0))))


def oracle_every_head(w, x, backward=True, workers=None):
    """The full oracle on every (b, h) head, one single-threaded oracle call per head on a thread pool (the
    oracle's C code runs without the GIL).  Arrays [B, H, N, d] (LSE [B, H, Nq]), like the GPU outputs."""
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def one(bh):
        b, h = bh
        s = {n: f64_head(x[n], b, h) for n in (("q", "k", "v", "do") if backward else ("q", "k", "v"))}
        o, lse = oracle.attn_fwd(s["q"], s["k"], s["v"], w.causal, w.scale)
        r = {"o": o[0, 0], "lse": lse[0, 0]}
        if backward:
            dq, dk, dv, _ = oracle.attn_bwd(s["q"], s["k"], s["v"], s["do"], w.causal, w.scale)
            r.update(dq=dq[0, 0], dk=dk[0, 0], dv=dv[0, 0])
        return r

    with concurrent.futures.ThreadPoolExecutor(max_workers=_workers(workers)) as ex:
        res = list(ex.map(one, heads))
    return {key: np.stack([r[key] for r in res]).reshape((w.B, w.H) + res[0][key].shape) for key in res[0]}


def oracle_one_head_split(w, x, b, h, workers=None):
    """Every output of one (long) head, its query rows split over a thread pool.  O, LSE and dQ are row-local
    (the row-sampled oracle calls on contiguous row ranges); dK and dV are sums over query rows (the
    column-sampled call over every key row, on query-row parts of about equal work, summed)."""
    s = {n: f64_head(x[n], b, h) for n in ("q", "k", "v", "do")}
    parts = query_parts(w.Nq, w.Nk, w.causal, _workers(workers))
    all_cols = np.arange(w.Nk, dtype=np.int64)

    def rows_part(r):
        rows = np.arange(r[0], r[1], dtype=np.int64)
        o, lse = oracle.attn_fwd_rows(s["q"], s["k"], s["v"], w.causal, w.scale, rows)
        dq, _ = oracle.attn_dq_rows(s["q"], s["k"], s["v"], s["do"], w.causal, w.scale, rows)
        return o, lse, dq

    def cols_part(r):
        return oracle.attn_dkdv_cols(s["q"], s["k"], s["v"], s["do"], w.causal, w.scale, all_cols, q_range=r)

    with concurrent.futures.ThreadPoolExecutor(max_workers=_workers(workers)) as ex:
        row_res = list(ex.map(rows_part, parts))
        col_res = list(ex.map(cols_part, parts))
    return {"o": np.concatenate([r[0] for r in row_res]), "lse": np.concatenate([r[1] for r in row_res]),
            "dq": np.concatenate([r[2] for r in row_res]), "dk": sum(c[0] for c in col_res),
            "dv": sum(c[1] for c in col_res)}
