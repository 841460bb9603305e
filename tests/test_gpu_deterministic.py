"""GPU parity and reproducibility of the deterministic dQ mode (attn_bwd_ex).

The deterministic backward must match the fp64 oracle like the atomic one,
give the same bits on every run, and give the atomic mode's dK and dV bit for
bit: the key/value-block kernel computes them the same way in both modes.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

from parity import check_grads, f64_head, heavy_cols, oracle_cols_threaded, oracle_every_head, rel_l2, sample_rows

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS

SHAPES = [
    (1, 2, 128, 128, 64, "fp16", False),
    (1, 2, 300, 300, 128, "bf16", True),
    (2, 1, 129, 257, 64, "bf16", False),
    (1, 1, 257, 129, 128, "fp16", True),
    (1, 2, 200, 700, 128, "bf16", "bottom_right"),
    (1, 1, 700, 300, 64, "bf16", "bottom_right"),   # rows that see no key, a query tile that sees none
    (1, 1, 1, 1, 128, "bf16", True),
    (3, 2, 384, 384, 128, "fp16", False),
]


def _grads(w, x, dq_mode, layout=None):
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    if layout is not None:
        q, k, v, do = layout(q), layout(k), layout(v), layout(do)
    o, lse = exattn.forward(q, k, v, w.causal, w.scale)
    dq, dk, dv = exattn.backward(q, k, v, o, do, lse, w.causal, w.scale, dq_mode=dq_mode)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    return dq, dk, dv


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}q{}k{}d{}{}{}".format(*s))
def test_deterministic_full_parity_and_repeatability(shape):
    w = workloads.custom(*shape)
    x = workloads.make_inputs(w)
    dq1, dk1, dv1 = _grads(w, x, "deterministic")
    dq2, dk2, dv2 = _grads(w, x, "deterministic")
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2), "not reproducible"
    dqa, dka, dva = _grads(w, x, "atomic")
    assert torch.equal(dk1, dka) and torch.equal(dv1, dva), "dK/dV differ between the dQ modes"
    # the same dS, summed in another order
    assert rel_l2(dq1.float().cpu().numpy(), dqa.float().cpu().numpy()) <= 2e-3
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale)
    got = {n: t.float().cpu().numpy() for n, t in (("dq", dq1), ("dk", dk1), ("dv", dv1))}
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, f"deterministic {w.name}")


def test_deterministic_strided_matches_contiguous():
    w = workloads.custom(2, 3, 300, 500, 128, "bf16", "bottom_right")
    x = workloads.make_inputs(w)
    a = _grads(w, x, "deterministic")
    bnhd = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)  # noqa: E731
    b = _grads(w, x, "deterministic", layout=bnhd)
    for ta, tb in zip(a, b):
        assert torch.equal(ta, tb)


@pytest.mark.parametrize("name", ["long8k_causal_bf16", "ctx32k_d128_causal_bf16"])
def test_deterministic_long_workloads_sampled(name):
    w = W[name]
    x = workloads.make_inputs(w)
    dq, dk, dv = _grads(w, x, "deterministic")
    dq, dk, dv = (t.float().cpu().numpy() for t in (dq, dk, dv))
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        bh = b * w.H + h
        rows = sample_rows(w.Nq, 32, 7 + bh)
        sel = lambda t: t[b:b + 1, h:h + 1]  # noqa: E731
        dq_r, _ = oracle.attn_dq_rows(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["do"]), w.causal, w.scale, rows)
        check_grads({"dq": dq[b, h, rows]}, {"dq": dq_r}, f"{name} head {bh} dQ rows")
        # the last key rows and those of the first key blocks (every query tile adds into them when causal)
        cols = np.array(sorted({w.Nk - 1, w.Nk - 100, w.Nk - 300, *heavy_cols(w.Nk).tolist()}), dtype=np.int64)
        xs = {n: f64_head(x[n], b, h) for n in ("q", "k", "v", "do")}

        def part(r):
            return oracle.attn_dkdv_cols(xs["q"], xs["k"], xs["v"], xs["do"], w.causal, w.scale, cols, q_range=r)

        dk_c, dv_c = oracle_cols_threaded(part, w.Nq, w.Nk, w.causal)
        check_grads({"dk": dk[b, h, cols], "dv": dv[b, h, cols]}, {"dk": dk_c, "dv": dv_c}, f"{name} head {bh}")


def test_deterministic_long_sequence_workload_every_element():
    """The deterministic mode on the long-sequence workload (B=1, H=12, N=8192, d=128, causal): every element
    of dQ, dK and dV of all twelve heads against the oracle (one oracle call per head on a thread pool)."""
    w = W["long8k_causal_bf16"]
    x = workloads.make_inputs(w)
    dq, dk, dv = (t.float().cpu().numpy() for t in _grads(w, x, "deterministic"))
    ref = oracle_every_head(w, x)
    for h in range(w.H):
        check_grads({"dq": dq[0, h], "dk": dk[0, h], "dv": dv[0, h]},
                    {k: ref[k][0, h] for k in ("dq", "dk", "dv")}, f"deterministic {w.name} head {h}")


def test_auto_mode_is_the_atomic_path():
    """ATTN_DQ_AUTO resolves to the reductions (measured faster on every shape tried)."""
    w = workloads.custom(1, 2, 256, 256, 64, "bf16", True)
    x = workloads.make_inputs(w)
    a = _grads(w, x, "auto")
    b = _grads(w, x, "atomic")
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert rel_l2(a[0].float().cpu().numpy(), b[0].float().cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("shape", [(16, 16, 2048, 128, False), (1, 4, 2048, 128, True), (4, 16, 8192, 128, True)],
                         ids=["nomask_256MiB_head_groups", "causal_heads_fastest", "causal_256MiB_head_groups"])
def test_atomic_matches_deterministic_in_both_launch_orders(shape):
    """The reductions' key blocks run heads fastest while the accumulator fits in half of L2 (a quarter with
    no mask), else in groups of a few heads (here 7 and 5, neither dividing the 256 and 64 heads, so the
    last group takes the remainder).  In each order dK and dV are the deterministic mode's bits (the
    key/value blocks compute them alike in both modes; the deterministic mode runs heads fastest) and dQ
    agrees within fp32 summation order; "auto" resolves to the reductions."""
    B, H, N, d, causal = shape
    assert exattn.auto_dq_mode(B, H, N, N, d, causal) == "atomic"
    want_g = {(16, 16, 2048, 128, False): 8, (1, 4, 2048, 128, True): 4, (4, 16, 8192, 128, True): 5}[shape]
    assert exattn.head_group(B, H, N, N, d, causal) == want_g  # this device's SM count and L2 size
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(B * H + N)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
    o, lse = exattn.forward(q, k, v, causal)
    auto = exattn.backward(q, k, v, o, do, lse, causal, dq_mode="auto")
    det = exattn.backward(q, k, v, o, do, lse, causal, dq_mode="deterministic")
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    assert torch.equal(auto[1], det[1]) and torch.equal(auto[2], det[2])
    assert rel_l2(auto[0].float().cpu().numpy(), det[0].float().cpu().numpy()) <= 1e-3
