"""GPU parity of the split-KV forward (attn_fwd_splitkv) against the fp64 CPU oracle.

Small shapes are compared on every output, over explicit slice counts that
leave some slices empty, masks of all three kinds and query tiles that see no
key.  The decoding workloads run at full size with the library's own slice
count, against the oracle on every row (one query per head) or on sampled rows
(64-query chunks).  With one slice the result must equal the plain forward bit
for bit (the same per-tile arithmetic, merged with weight 1).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

from parity import check_fwd, sample_rows

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


def _run(w, x, num_splits, layout=None):
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    if layout is not None:
        q, k, v = layout(q), layout(k), layout(v)
    o, lse = exattn.forward_splitkv(q, k, v, w.causal, w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    return o, lse


SMALL = [
    # (B, H, Nq, Nk, d, dtype, causal, num_splits)
    (1, 2, 1, 1000, 128, "bf16", False, 4),
    (2, 1, 64, 1000, 64, "fp16", "bottom_right", 3),
    (1, 1, 200, 700, 128, "bf16", True, 5),           # top-left: the second query tile sees one more tile
    (1, 1, 1, 200, 64, "bf16", False, 8),             # 2 key tiles over 8 slices: 6 slices are empty
    (1, 1, 300, 100, 128, "fp16", "bottom_right", 2), # rows 0..199 see no key; query tile 0 sees none
    (3, 2, 17, 4099, 128, "bf16", "bottom_right", 7), # ragged key tail inside a slice
    (1, 3, 1, 129, 64, "fp16", False, 1),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}q{}k{}d{}{}{}s{}".format(*s))
def test_splitkv_small_full_parity(shape):
    B, H, Nq, Nk, d, dt, causal, splits = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal)
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _run(w, x, splits)
    ref_o, ref_lse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    check_fwd(w, o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, f"{w.name} splits={splits}")


@pytest.mark.parametrize("shape", [(1, 2, 1, 1000, 128, "bf16", False), (2, 3, 200, 700, 64, "fp16", True),
                                   (1, 1, 64, 513, 128, "bf16", "bottom_right")],
                         ids=lambda s: "B{}H{}q{}k{}d{}{}{}".format(*s))
def test_one_slice_equals_plain_forward(shape):
    w = workloads.custom(*shape)
    x = workloads.make_inputs(w, with_grad_out=False)
    o_s, lse_s = _run(w, x, 1)
    dev = torch.device("cuda")
    o_p, lse_p = exattn.forward(*(x[n].to(dev) for n in ("q", "k", "v")), w.causal, w.scale)
    assert torch.equal(o_s, o_p) and torch.equal(lse_s, lse_p)


def test_splitkv_strided_cache_matches_contiguous():
    """A [B, N, H, d] key/value cache gives the same bits as the contiguous layout."""
    w = workloads.custom(2, 4, 3, 3000, 128, "bf16", "bottom_right")
    x = workloads.make_inputs(w, with_grad_out=False)
    o_c, lse_c = _run(w, x, 5)
    bnhd = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)  # noqa: E731
    o_s, lse_s = _run(w, x, 5, layout=bnhd)
    assert torch.equal(o_s, o_c) and torch.equal(lse_s, lse_c)


def test_splitkv_outputs_written_everywhere():
    w = workloads.custom(2, 3, 70, 2000, 64, "bf16", "bottom_right")
    x = workloads.make_inputs(w, with_grad_out=False)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.Nq), float("nan"), device=dev)
    ws = torch.full((exattn.splitkv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, 6),), 0xFF, dtype=torch.uint8,
                    device=dev)
    assert exattn.fwd_splitkv_raw(q, k, v, o, lse, w.causal, w.scale, 6, ws) == 0
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def _head(x, name, b, h):
    return x[name][b:b + 1, h:h + 1]


def test_decode_workload_every_row():
    """One new query per head over a 32k cache: every head against the oracle (one head per call)."""
    w = W["decode_q1_kv32k_d128_bf16"]
    assert exattn.splitkv_num_splits(w.B, w.H, w.Nq, w.Nk, w.d) > 1
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _run(w, x, 0)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(w.B):
        for h in range(w.H):
            ref_o, ref_lse = oracle.attn_fwd(_head(x, "q", b, h), _head(x, "k", b, h), _head(x, "v", b, h),
                                             w.causal, w.scale)
            check_fwd(w, o[b, h], lse[b, h], ref_o[0, 0], ref_lse[0, 0], f"{w.name} head {b * w.H + h}")


def test_chunk_workload_sampled_rows():
    w = W["chunk_q64_kv16k_d64_fp16"]
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _run(w, x, 0)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1), (1, 7)]:
        rows = sample_rows(w.Nq, 16, 100 + b * w.H + h)
        o_r, lse_r = oracle.attn_fwd_rows(_head(x, "q", b, h), _head(x, "k", b, h), _head(x, "v", b, h),
                                          w.causal, w.scale, rows)
        check_fwd(w, o[b, h, rows], lse[b, h, rows], o_r, lse_r, f"{w.name} head {b * w.H + h}")
