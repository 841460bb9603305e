"""The C ABI on caller streams: CUDA-graph capture, non-default streams, and a pipelined loop.

Every entry point takes a stream, launches only on it, allocates nothing and
never synchronises, so its calls can be captured into a CUDA graph and mixed
with copies on other streams.  These tests check exactly that against the same
calls made eagerly on one stream: the results must be the same bits (the
forward and the deterministic-dQ backward are deterministic), and one case is
also checked against the fp64 oracle.
"""
import pytest
import torch

import oracle
from exact_head_attention_gb300 import exattn, workloads

from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _inputs(shape, index):
    w = workloads.custom(*shape, index=index)
    x = workloads.make_inputs(w)
    return w, {n: x[n].to(DEV) for n in ("q", "k", "v", "do")}, x


def _buffers(d):
    q = d["q"]
    B, H, Nq, _ = q.shape
    return {
        "o": torch.empty_like(q), "lse": torch.empty((B, H, Nq), dtype=torch.float32, device=DEV),
        "dq": torch.empty_like(q), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
        "ws": torch.empty(exattn.workspace_size(B, H, Nq, q.shape[3]), dtype=torch.uint8, device=DEV),
    }


def _step(w, d, b, stream):
    """Forward then backward (deterministic dQ) through the raw C-ABI calls on `stream`."""
    s1 = exattn.fwd_raw(d["q"], d["k"], d["v"], b["o"], b["lse"], w.causal, w.scale, stream=stream)
    s2 = exattn.bwd_ex_raw(d["q"], d["k"], d["v"], b["o"], d["do"], b["lse"], b["dq"], b["dk"], b["dv"], w.causal,
                           w.scale, "deterministic", b["ws"], stream=stream)
    assert s1 == 0 and s2 == 0, exattn.last_error()


def _snapshot(b):
    return {n: b[n].clone() for n in ("o", "lse", "dq", "dk", "dv")}


def _assert_same(got, want, what):
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(got[n], want[n]), f"{what}: {n} differs"


@pytest.mark.parametrize("shape", [(1, 2, 300, 300, 128, "bf16", True), (2, 1, 129, 257, 64, "fp16", "bottom_right")],
                         ids=str)
def test_graph_capture_replays_the_eager_results(shape):
    w, d, x = _inputs(shape, 60)
    b = _buffers(d)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        _step(w, d, b, side)
    side.synchronize()
    eager = _snapshot(b)
    ro, rlse = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    check_fwd(w, eager["o"].float().cpu().numpy(), eager["lse"].cpu().numpy(), ro, rlse, f"{w.name} eager")

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        _step(w, d, b, side)
    for n in ("o", "lse", "dq", "dk", "dv"):
        b[n].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    _assert_same(_snapshot(b), eager, "first replay")

    # New inputs copied into the captured buffers: the replay must compute on them.
    w2, d2, x2 = _inputs(shape, 61)
    for n in ("q", "k", "v", "do"):
        d[n].copy_(d2[n])
    g.replay()
    torch.cuda.synchronize()
    replay2 = _snapshot(b)
    b2 = _buffers(d2)
    _step(w2, d2, b2, torch.cuda.current_stream())
    torch.cuda.synchronize()
    _assert_same(replay2, _snapshot(b2), "replay on new inputs")
    rdq, rdk, rdv, _ = oracle.attn_bwd(x2["q"], x2["k"], x2["v"], x2["do"], w2.causal, w2.scale)
    check_grads({n: replay2[n].float().cpu().numpy() for n in ("dq", "dk", "dv")}, {"dq": rdq, "dk": rdk, "dv": rdv},
                f"{w2.name} replay")


def test_graph_capture_of_the_splitkv_forward():
    w, d, _ = _inputs((2, 3, 1, 3000, 128, "bf16", "bottom_right"), 62)
    q, k, v = d["q"], d["k"], d["v"]
    splits = 4
    ws = torch.empty(exattn.splitkv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, splits), dtype=torch.uint8, device=DEV)
    o, lse = torch.empty_like(q), torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=DEV)
    side = torch.cuda.Stream()
    assert exattn.fwd_splitkv_raw(q, k, v, o, lse, w.causal, w.scale, splits, ws, stream=side) == 0
    side.synchronize()
    o_eager, lse_eager = o.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        assert exattn.fwd_splitkv_raw(q, k, v, o, lse, w.causal, w.scale, splits, ws, stream=side) == 0
    o.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)


def test_two_side_streams_while_the_default_stream_is_busy():
    problems = [_inputs((1, 2, 384, 384, 128, "bf16", True), 63), _inputs((2, 2, 200, 333, 64, "fp16", False), 64)]
    eager = []
    for w, d, _ in problems:
        b = _buffers(d)
        _step(w, d, b, torch.cuda.current_stream())
        torch.cuda.synchronize()
        eager.append(_snapshot(b))

    bufs = [_buffers(d) for _, d, _ in problems]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    filler = torch.empty(1 << 28, dtype=torch.uint8, device=DEV)
    filler.fill_(1)  # keeps the default stream busy while the side streams launch
    for (w, d, _), b, s in zip(problems, bufs, streams):
        with torch.cuda.stream(s):
            _step(w, d, b, s)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    for i, b in enumerate(bufs):
        _assert_same(_snapshot(b), eager[i], f"side stream {i}")


def test_pipelined_steps_over_three_streams():
    """Two device buffer sets, copy-in / compute / copy-out streams (the end-to-end loop bench.py times)."""
    shape = (1, 2, 256, 256, 128, "bf16", True)
    steps = [workloads.make_inputs(workloads.custom(*shape, index=70 + i)) for i in range(5)]
    w = workloads.custom(*shape, index=70)
    host_in = [{n: x[n].pin_memory() for n in ("q", "k", "v", "do")} for x in steps]
    sets = []
    for _ in range(2):
        d = {n: torch.empty_like(t, device=DEV) for n, t in host_in[0].items()}
        sets.append((d, _buffers(d)))
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in sets[0][1].items() if n != "ws"}
                for _ in steps]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    cmp_done, out_done = [], []
    for i in range(len(steps)):
        d, b = sets[i % 2]
        if i >= 2:
            s_in.wait_event(cmp_done[i - 2])
        with torch.cuda.stream(s_in):
            for n in d:
                d[n].copy_(host_in[i][n], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(s_in)
        s_cmp.wait_event(ev)
        if i >= 2:
            s_cmp.wait_event(out_done[i - 2])
        _step(w, d, b, s_cmp)
        cmp_done.append(torch.cuda.Event())
        cmp_done[-1].record(s_cmp)
        s_out.wait_event(cmp_done[-1])
        with torch.cuda.stream(s_out):
            for n, t in host_out[i].items():
                t.copy_(b[n], non_blocking=True)
        out_done.append(torch.cuda.Event())
        out_done[-1].record(s_out)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    for i, x in enumerate(steps):
        d = {n: x[n].to(DEV) for n in ("q", "k", "v", "do")}
        b = _buffers(d)
        _step(w, d, b, torch.cuda.current_stream())
        torch.cuda.synchronize()
        _assert_same({n: t.to(DEV) for n, t in host_out[i].items()}, _snapshot(b), f"step {i}")
