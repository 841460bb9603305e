"""Seeded random shapes through every attention entry point, against the fp64 oracle.

Each case draws B, H, Nq, Nk (1 to 700, so single rows, ragged tails and
several tiles all occur), d, dtype, mask and layout from a fixed seed, and
checks the forward, the backward in both dQ modes and the split-KV forward
with a random slice count against the oracle at the usual tolerances.
"""
import random

import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu

MASKS = [False, True, "bottom_right"]


def _case(seed):
    r = random.Random(seed)
    B, H = r.randint(1, 3), r.randint(1, 3)
    Nq = r.choice([1, r.randint(2, 130), r.randint(131, 700)])
    Nk = r.choice([1, r.randint(2, 130), r.randint(131, 700)])
    d = r.choice([64, 128])
    dt = r.choice(["bf16", "fp16"])
    causal = r.choice(MASKS)
    layout = r.choice(["contiguous", "bnhd"])
    splits = r.randint(1, 6)
    return B, H, Nq, Nk, d, dt, causal, layout, splits


def _bnhd(t):
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(seed):
    B, H, Nq, Nk, d, dt, causal, layout, splits = _case(seed)
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal, index=20 + seed)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    if layout == "bnhd":
        q, k, v, do = _bnhd(q), _bnhd(k), _bnhd(v), _bnhd(do)
    what = f"seed {seed}: B{B} H{H} q{Nq} k{Nk} d{d} {dt} mask={causal} {layout}"

    o, lse = exattn.forward(q, k, v, causal, w.scale)
    ro, rlse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    check_fwd(w, o.float().cpu().numpy(), lse.cpu().numpy(), ro, rlse, what)

    rdq, rdk, rdv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
    for mode in ("atomic", "deterministic"):
        dq, dk, dv = exattn.backward(q, k, v, o, do, lse, causal, w.scale, dq_mode=mode)
        got = {n: t.float().cpu().numpy() for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
        check_grads(got, {"dq": rdq, "dk": rdk, "dv": rdv}, f"{what} {mode}")

    os_, lses = exattn.forward_splitkv(q, k, v, causal, w.scale, num_splits=splits)
    check_fwd(w, os_.float().cpu().numpy(), lses.cpu().numpy(), ro, rlse, f"{what} splitkv {splits}")
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
