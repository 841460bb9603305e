"""GPU parity of the bottom-right causal mask and of strided layouts ([B, N, H, d]
storage, padded rows, mixed layouts) against the fp64 CPU oracle.

Bottom-right shapes cover a diagonal offset that is not a tile multiple, Nq < Nk
and Nq > Nk (rows that see no key, and a whole query block that sees none), a
single query, and the square case (identical to top-left).  Strided runs must
also agree bit for bit with the contiguous path on O, LSE, dK and dV: the
kernels are the same, and only the tensor maps differ.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

from parity import check_fwd, check_grads, run_gpu

pytestmark = pytest.mark.gpu

BOTTOM_RIGHT = [
    (1, 2, 200, 700, 128, "bf16"),   # offset 500: not a multiple of the 128-row tile
    (2, 1, 64, 1000, 64, "fp16"),    # a chunk of 64 new queries over a long cache
    (1, 1, 700, 300, 64, "bf16"),    # rows 0..399 see no key; the first 256-row block sees none at all
    (1, 2, 513, 129, 128, "fp16"),   # Nq > Nk with ragged tails
    (1, 1, 1, 333, 128, "bf16"),     # one query sees every key
    (1, 2, 384, 384, 64, "bf16"),    # square: the same mask as top-left
]


@pytest.mark.parametrize("shape", BOTTOM_RIGHT, ids=lambda s: "B{}H{}q{}k{}d{}{}".format(*s))
def test_bottom_right_full_parity(shape):
    B, H, Nq, Nk, d, dt = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, "bottom_right")
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], 2, w.scale)
    check_fwd(w, got["o"], got["lse"], o, lse, w.name)
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], 2, w.scale)
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, w.name)
    if Nq > Nk:
        assert (got["dq"][:, :, : Nq - Nk] == 0).all(), "dQ of rows without keys is not 0"


def test_bottom_right_square_equals_top_left():
    w = workloads.custom(1, 2, 384, 384, 128, "bf16", True)
    x = workloads.make_inputs(w)
    a = run_gpu(w, x, backward=False)
    b = run_gpu(w.replace(causal="bottom_right"), x, backward=False)
    np.testing.assert_array_equal(a["o"], b["o"])
    np.testing.assert_array_equal(a["lse"], b["lse"])


def _bnhd(t):
    """The same values stored as [B, N, H, d] (rows of [S, H*D]) and viewed as [B, H, N, d]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _padded_rows(t, pad=64):
    """The same values in a [B, H, N, d + pad] buffer, viewed as [B, H, N, d] (row stride d + pad)."""
    buf = torch.zeros(*t.shape[:-1], t.shape[-1] + pad, dtype=t.dtype, device=t.device)
    buf[..., : t.shape[-1]] = t
    return buf[..., : t.shape[-1]]


LAYOUTS = {
    "bnhd": (_bnhd, _bnhd, _bnhd),
    "q_bnhd_kv_contiguous": (_bnhd, lambda t: t, _bnhd),
    "padded_rows": (_padded_rows, _padded_rows, lambda t: t),
}


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("shape", [
    (2, 3, 300, 300, 128, "bf16", True),
    (1, 4, 129, 517, 64, "fp16", False),
    (2, 2, 200, 700, 128, "bf16", "bottom_right"),
], ids=lambda s: "B{}H{}q{}k{}d{}{}{}".format(*s))
def test_strided_layouts_match_contiguous_and_oracle(layout, shape):
    B, H, Nq, Nk, d, dt, causal = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o_c, lse_c = exattn.forward(q, k, v, causal, w.scale)
    dq_c, dk_c, dv_c = exattn.backward(q, k, v, o_c, do, lse_c, causal, w.scale)

    fq, fkv, fo = LAYOUTS[layout]
    qs, ks, vs, dos = fq(q), fkv(k), fkv(v), fo(do)
    assert not (qs.is_contiguous() and ks.is_contiguous())
    o_s, lse_s = exattn.forward(qs, ks, vs, causal, w.scale)
    o_in = fo(o_s.contiguous())  # O in the dO layout, so that the backward sees a strided O as well
    dq_s, dk_s, dv_s = exattn.backward(qs, ks, vs, o_in, dos, lse_s, causal, w.scale)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0

    assert torch.equal(o_s, o_c) and torch.equal(lse_s, lse_c), "strided forward differs from contiguous"
    assert torch.equal(dk_s, dk_c) and torch.equal(dv_s, dv_c), "strided dK/dV differ from contiguous"
    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    check_fwd(w, o_s.float().cpu().numpy(), lse_s.cpu().numpy(), o, lse, f"{layout} {w.name}")
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
    got = {n: t.float().cpu().numpy() for n, t in (("dq", dq_s), ("dk", dk_s), ("dv", dv_s))}
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, f"{layout} {w.name}")
    if layout == "bnhd":  # dense views: the gradients take the inputs' strides
        assert dq_s.stride() == qs.stride() and dk_s.stride() == ks.stride()
    del dq_c


def test_strided_writes_stay_inside_the_view():
    """Padding columns between strided rows keep their sentinel values."""
    w = workloads.custom(1, 2, 200, 150, 64, "bf16", True)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o_buf = torch.full((1, 2, 200, 128), 7.0, dtype=q.dtype, device=dev)
    o = o_buf[..., :64]
    lse = torch.empty((1, 2, 200), dtype=torch.float32, device=dev)
    assert exattn.fwd_strided_raw(q, k, v, o, lse, True, w.scale) == 0
    dq_buf, dk_buf, dv_buf = (torch.full((1, 2, n, 128), 7.0, dtype=q.dtype, device=dev) for n in (200, 150, 150))
    dq, dk, dv = dq_buf[..., :64], dk_buf[..., :64], dv_buf[..., :64]
    ws = torch.empty(exattn.workspace_size(1, 2, 200, 64), dtype=torch.uint8, device=dev)
    assert exattn.bwd_strided_raw(q, k, v, o, do, lse, dq, dk, dv, True, w.scale, ws) == 0
    torch.cuda.synchronize()
    for buf in (o_buf, dq_buf, dk_buf, dv_buf):
        assert (buf[..., 64:] == 7.0).all()
    ref_o, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], True, w.scale)
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= 1e-2
