"""GPU parity of the attention-KL forward and backward (attn_kl_fwd, attn_kl_bwd, attn_kl_bwd_ex) against the
fp64 oracle.

The backward is checked in both dQ modes: "deterministic" (two launches, the same bits on every run) and
"atomic" (one pass over key tiles; dK is the same bits on every run, dQ's fp32 summation order is not).

Tolerances: KL, LSE1 and LSE2 max-abs <= 1e-3 (the LSE bound of the attention
path; KL is a sum of an fp32 mean logit difference and two LSEs, each good to
about 1e-5 here), dQ and dK relative L2 <= 2e-2 (the attention gradients'
bound: dS is rounded to the 16-bit input type before the gradient products).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

import concurrent.futures
import os

from parity import f64_head, heavy_cols, oracle_cols_threaded, rel_l2, sample_rows

pytestmark = pytest.mark.gpu

KL_TOL = 1e-3
LSE_TOL = 1e-3
GRAD_TOL = 2e-2

SHAPES = [
    (1, 2, 128, 128, 64, "fp16", False),
    (1, 2, 300, 300, 128, "bf16", True),
    (2, 1, 129, 257, 64, "bf16", False),
    (1, 2, 200, 700, 128, "bf16", "bottom_right"),
    (1, 1, 500, 200, 64, "fp16", "bottom_right"),  # rows without keys, a query tile without keys
    (1, 1, 1, 1, 128, "bf16", True),
    (2, 3, 384, 384, 128, "bf16", True),
]


def _dev(x):
    dev = torch.device("cuda")
    return {k: v.to(dev) for k, v in x.items()}


def _check_fwd(kl, l1, l2, ref, what):
    rkl, rl1, rl2 = ref
    empty = np.isneginf(rl1)
    assert np.isneginf(l1[empty]).all() and np.isneginf(l2[empty]).all() and (kl[empty] == 0).all(), what
    for got, want, tol, name in ((kl, rkl, KL_TOL, "KL"), (l1, rl1, LSE_TOL, "LSE1"), (l2, rl2, LSE_TOL, "LSE2")):
        g, w = got[~empty], want[~empty]
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        err = float(np.abs(g - w).max()) if g.size else 0.0
        assert err <= tol, f"{what}: {name} max-abs {err:.3e} > {tol}"


MODES = ("deterministic", "atomic")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}q{}k{}d{}{}{}".format(*s))
def test_kl_small_full_parity(shape, mode):
    w = workloads.custom(*shape)
    x = workloads.make_kl_inputs(w)
    d = _dev(x)
    kl, l1, l2 = exattn.kl_forward(d["q1"], d["k1"], d["q2"], d["k2"], w.causal, w.scale)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    ref = oracle.kl_fwd(x["q1"], x["k1"], x["q2"], x["k2"], w.causal, w.scale)
    _check_fwd(kl.cpu().numpy(), l1.cpu().numpy(), l2.cpu().numpy(), ref, w.name)
    for train, setting in (("student", 1), ("teacher", 2)):
        args = (d["q1"], d["k1"], d["q2"], d["k2"], kl, l1, l2, d["g"], train, w.causal, w.scale)
        dq, dk = exattn.kl_backward(*args, dq_mode=mode)
        dq2, dk2 = exattn.kl_backward(*args, dq_mode=mode)
        torch.cuda.synchronize()
        assert exattn.check_device_error() == 0
        assert torch.equal(dk, dk2), "dK not reproducible"
        if mode == "deterministic":
            assert torch.equal(dq, dq2), "dQ not reproducible"
        rdq, rdk = oracle.kl_bwd(x["q1"], x["k1"], x["q2"], x["k2"], x["g"], setting, w.causal, w.scale)
        for name, got, want in (("dQ", dq, rdq), ("dK", dk, rdk)):
            got = got.float().cpu().numpy()
            assert np.isfinite(got).all(), f"{w.name} {train}: non-finite {name}"
            err = rel_l2(got, want)
            assert err <= GRAD_TOL, f"{w.name} {train}: {name} rel-L2 {err:.3e}"


@pytest.mark.parametrize("mode", MODES)
def test_kl_identical_distributions(mode):
    """Teacher == student: KL is 0 up to rounding and the student's gradient vanishes."""
    w = workloads.custom(1, 2, 256, 256, 128, "bf16", True)
    x = workloads.make_kl_inputs(w)
    d = _dev(x)
    kl, l1, l2 = exattn.kl_forward(d["q1"], d["k1"], d["q1"], d["k1"], True)
    assert torch.equal(l1, l2)
    assert kl.abs().max().item() <= 1e-5
    dq, dk = exattn.kl_backward(d["q1"], d["k1"], d["q1"], d["k1"], kl, l1, l2, d["g"], "student", True, dq_mode=mode)
    assert dq.float().abs().max().item() <= 1e-3 and dk.float().abs().max().item() <= 1e-3


def test_kl_autograd_routes_gradients():
    w = workloads.custom(1, 2, 200, 200, 64, "bf16", "bottom_right")
    x = workloads.make_kl_inputs(w)
    d = {k: v.clone().requires_grad_(k != "g") for k, v in _dev(x).items()}
    kl = exattn.attention_kl(d["q1"], d["k1"], d["q2"], d["k2"], w.causal, train="student")
    (kl * d["g"]).sum().backward()
    assert d["q1"].grad is None and d["k1"].grad is None
    rdq, rdk = oracle.kl_bwd(x["q1"], x["k1"], x["q2"], x["k2"], x["g"], 1, w.causal, w.scale)
    assert rel_l2(d["q2"].grad.float().cpu().numpy(), rdq) <= GRAD_TOL
    assert rel_l2(d["k2"].grad.float().cpu().numpy(), rdk) <= GRAD_TOL


@pytest.mark.parametrize("mode,shape", [(m, None) for m in MODES] + [("atomic", (4, 16, 8192, 8192, 128, "bf16", True))],
                         ids=lambda v: v if isinstance(v, str) else ("B{}H{}q{}k{}d{}{}{}".format(*v) if v else "kl8k"))
def test_kl_workload_full_size_sampled(mode, shape):
    """The 8k workload, and 64 heads whose 256 MiB dQ accumulator makes the one pass launch its key tiles
    in groups of a few heads."""
    w = workloads.WORKLOADS["kl8k_causal_bf16"] if shape is None else workloads.custom(*shape, index=33)
    x = workloads.make_kl_inputs(w)
    d = _dev(x)
    kl, l1, l2 = exattn.kl_forward(d["q1"], d["k1"], d["q2"], d["k2"], w.causal, w.scale)
    grads = {t: exattn.kl_backward(d["q1"], d["k1"], d["q2"], d["k2"], kl, l1, l2, d["g"], t, w.causal, w.scale,
                                   dq_mode=mode)
             for t in ("student", "teacher")}
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    kl, l1, l2 = kl.cpu().numpy(), l1.cpu().numpy(), l2.cpu().numpy()
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        sel = lambda t: t[b:b + 1, h:h + 1]  # noqa: E731
        args = (sel(x["q1"]), sel(x["k1"]), sel(x["q2"]), sel(x["k2"]))
        rows = sample_rows(w.Nq, 48, 11 + h)
        ref = oracle.kl_fwd_rows(*args, w.causal, w.scale, rows)
        _check_fwd(kl[b, h, rows], l1[b, h, rows], l2[b, h, rows], ref, f"{w.name} head {h}")
        # the last key rows and those of the first key tiles (every query tile adds into them when causal)
        cols = np.array(sorted({w.Nk - 1, w.Nk - 77, w.Nk - 300, *heavy_cols(w.Nk).tolist()}), dtype=np.int64)
        a64 = tuple(f64_head(x[n], b, h) for n in ("q1", "k1", "q2", "k2"))
        g64 = f64_head(x["g"], b, h)
        for train, setting in (("student", 1), ("teacher", 2)):
            dq, dk = (t.float().cpu().numpy() for t in grads[train])
            rq = oracle.kl_dq_rows(*args, sel(x["g"]), setting, w.causal, w.scale, rows[:24])
            assert rel_l2(dq[b, h, rows[:24]], rq) <= GRAD_TOL, f"{train} dQ rows head {h}"

            def part(r, setting=setting):
                return oracle.kl_dk_cols(*a64, g64, setting, w.causal, w.scale, cols, q_range=r)

            rk = oracle_cols_threaded(part, w.Nq, w.Nk, w.causal)
            assert rel_l2(dk[b, h, cols], rk) <= GRAD_TOL, f"{train} dK rows {cols.tolist()} head {h}"


def _kl_oracle_every_head(w, x):
    """The KL oracle (forward, both backward settings) on every head, one head per thread."""
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def one(bh):
        b, h = bh
        a = tuple(f64_head(x[n], b, h) for n in ("q1", "k1", "q2", "k2"))
        g = f64_head(x["g"], b, h)
        out = dict(zip(("kl", "l1", "l2"), (t[0, 0] for t in oracle.kl_fwd(*a, w.causal, w.scale))))
        for setting in (1, 2):
            dq, dk = oracle.kl_bwd(*a, g, setting, w.causal, w.scale)
            out[f"dq{setting}"], out[f"dk{setting}"] = dq[0, 0], dk[0, 0]
        return out

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, len(os.sched_getaffinity(0))))) as ex:
        res = list(ex.map(one, heads))
    return {k: np.stack([r[k] for r in res]).reshape((w.B, w.H) + res[0][k].shape) for k in res[0]}


def test_kl_workload_every_element():
    """The KL workload (B=1, H=12, N=8192, d=128, causal) in full: KL, LSE1, LSE2 and, in both dQ modes and
    both settings, every element of dQ and dK of all twelve heads against the oracle (one head per
    thread)."""
    w = workloads.WORKLOADS["kl8k_causal_bf16"]
    x = workloads.make_kl_inputs(w)
    d = _dev(x)
    kl, l1, l2 = exattn.kl_forward(d["q1"], d["k1"], d["q2"], d["k2"], w.causal, w.scale)
    grads = {(m, t): exattn.kl_backward(d["q1"], d["k1"], d["q2"], d["k2"], kl, l1, l2, d["g"], t, w.causal,
                                         w.scale, dq_mode=m)
             for m in MODES for t in ("student", "teacher")}
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    ref = _kl_oracle_every_head(w, x)
    _check_fwd(kl.cpu().numpy(), l1.cpu().numpy(), l2.cpu().numpy(), (ref["kl"], ref["l1"], ref["l2"]), w.name)
    for (m, t), (dq, dk) in grads.items():
        setting = 1 if t == "student" else 2
        dq, dk = dq.float().cpu().numpy(), dk.float().cpu().numpy()
        for h in range(w.H):
            assert rel_l2(dq[0, h], ref[f"dq{setting}"][0, h]) <= GRAD_TOL, f"{m} {t} dQ head {h}"
            assert rel_l2(dk[0, h], ref[f"dk{setting}"][0, h]) <= GRAD_TOL, f"{m} {t} dK head {h}"


@pytest.mark.parametrize("shape,splits", [
    ((2, 3, 1, 3000, 128, "bf16", "bottom_right"), 4),    # one query per head (decoding)
    ((1, 2, 64, 2000, 64, "fp16", "bottom_right"), 3),
    ((1, 1, 200, 700, 128, "bf16", True), 5),            # top-left: the second query tile sees one more tile
    ((1, 1, 1, 200, 64, "bf16", False), 8),              # two key tiles over eight slices: empty slices
    ((1, 1, 300, 100, 128, "fp16", "bottom_right"), 2),  # rows and a query tile without keys
    ((2, 2, 5, 4099, 64, "bf16", False), 0),             # the library's slice count
], ids=lambda v: str(v))
def test_kl_splitkv_parity(shape, splits):
    w = workloads.custom(*shape)
    x = workloads.make_kl_inputs(w)
    d = _dev(x)
    kl, l1, l2 = exattn.kl_forward_splitkv(d["q1"], d["k1"], d["q2"], d["k2"], w.causal, w.scale, num_splits=splits)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    ref = oracle.kl_fwd(x["q1"], x["k1"], x["q2"], x["k2"], w.causal, w.scale)
    _check_fwd(kl.cpu().numpy(), l1.cpu().numpy(), l2.cpu().numpy(), ref, f"{w.name} splits={splits}")
