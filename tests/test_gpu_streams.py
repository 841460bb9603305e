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


def _atomic_bwd(w, d, b, stream):
    s = exattn.bwd_raw(d["q"], d["k"], d["v"], b["o"], d["do"], b["lse"], b["dq"], b["dk"], b["dv"], w.causal,
                       w.scale, b["ws"], stream=stream)
    assert s == 0, exattn.last_error()


def _close_dq(got, want, what):
    err = (got.double() - want.double()).norm() / want.double().norm().clamp_min(1e-30)
    assert err < 1e-4, f"{what}: dQ rel-L2 {float(err):.2e}"


@pytest.mark.parametrize("shape", [(1, 4, 1024, 1024, 128, "bf16", True), (2, 2, 700, 500, 64, "fp16", False)],
                         ids=str)
def test_back_to_back_backwards_share_one_workspace(shape):
    """The backward's three kernels are dependent launches: the next call's preprocess zeroes the shared
    workspace only after the previous call's conversion has read it.  Two backward calls queued back to
    back on one stream with one workspace must give what each gives alone (dK, dV bitwise; dQ within
    fp32 summation order)."""
    stream = torch.cuda.current_stream()
    probs = [_inputs(shape, 80 + i) for i in range(2)]
    bufs = [_buffers(d) for _, d, _ in probs]
    alone = []
    for (w, d, _), b in zip(probs, bufs):
        assert exattn.fwd_raw(d["q"], d["k"], d["v"], b["o"], b["lse"], w.causal, w.scale, stream=stream) == 0
        _atomic_bwd(w, d, b, stream)
        torch.cuda.synchronize()
        alone.append(_snapshot(b))
    shared = bufs[0]["ws"]
    for b in bufs:
        b["ws"] = shared
        for n in ("dq", "dk", "dv"):
            b[n].zero_()
    for (w, d, _), b in zip(probs, bufs):
        _atomic_bwd(w, d, b, stream)
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    for i, b in enumerate(bufs):
        assert torch.equal(b["dk"], alone[i]["dk"]) and torch.equal(b["dv"], alone[i]["dv"]), f"call {i}"
        _close_dq(b["dq"], alone[i]["dq"], f"call {i}")


def test_input_written_by_the_kernel_just_before_the_backward():
    """dO written on the stream by a device copy right before the backward call: the preprocess and the
    main kernel (dependent launches) must see the new values, not the old ones."""
    shape = (1, 4, 1024, 1024, 128, "bf16", True)
    stream = torch.cuda.current_stream()
    w, d, _ = _inputs(shape, 90)
    _, d2, _ = _inputs(shape, 91)
    b = _buffers(d)
    assert exattn.fwd_raw(d["q"], d["k"], d["v"], b["o"], b["lse"], w.causal, w.scale, stream=stream) == 0
    ref = {"do": d2["do"]}
    ref.update({n: d[n] for n in ("q", "k", "v")})
    b_ref = _buffers(d)
    b_ref["o"].copy_(b["o"])
    b_ref["lse"].copy_(b["lse"])
    _atomic_bwd(w, ref, b_ref, stream)
    torch.cuda.synchronize()
    for _ in range(3):
        d["do"].copy_(d2["do"].flip(-1))  # something else first
        d["do"].copy_(d2["do"])           # the values the backward must read, written just before it
        _atomic_bwd(w, d, b, stream)
        torch.cuda.synchronize()
        assert torch.equal(b["dk"], b_ref["dk"]) and torch.equal(b["dv"], b_ref["dv"])
        _close_dq(b["dq"], b_ref["dq"], "dQ")
