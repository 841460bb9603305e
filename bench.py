#!/usr/bin/env python3
"""Throughput benchmark: exact fused attention, forward + backward, on GB300.

One step = attn_fwd, then the backward's three C-ABI steps (attn_bwd_preprocess,
attn_bwd_kv_blocks, attn_bwd_dq_convert -- together exactly attn_bwd) over one
batch of the synthetic workload.  The default workload is the long-sequence,
small-batch attention layer: B=1, H=12, Nq=Nk=8192, d=128, bf16, causal.

FLOPs per step follow the metric's convention: forward 4*B*H*Nq*Nk*d, backward
2.5x that, both halved when causal.

Timing: W untimed warm-up steps, then K timed steps; between timed steps a
256 MiB buffer is written (L2 flush) outside the timed events; every launch is
bracketed by CUDA events on the launching stream; ms_per_step is the median
of the per-step device times, max over ranks (the mean is reported beside
it).  With N > 1 (torchrun) every rank runs an independent replica of the
workload (no collective on the data path).

--impl reference times the CPU oracle (the plain fp64 definition) on the host
cores instead, on bounded samples of the same workload.

--workload kl8k_causal_bf16 times the attention KL divergence instead: one
step is attn_kl_fwd and attn_kl_bwd (the student trained), at 2 + 4 tile
products per (query tile, key tile) pair (the backward recomputes both score
tiles in each of its two kernels: 6 executed).

--workload NAME picks another workload.  A decoding workload (few queries over a
long key/value cache) times one split-KV forward (attn_fwd_splitkv: the slice
kernel and the merge kernel) per step and reports the bandwidth of its
algorithmic bytes (Q, K, V read once, O and LSE written once) against the
measured HBM copy bandwidth.

Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOPS (causal-adjusted) and % of GB300 BF16 tensor peak"
FALLBACK_BF16_TFLOPS = 1900.0
SPEC_BF16_TFLOPS = 2500.0  # GB300 dense bf16 tensor rate as specified (no sparsity), for context beside the measured peak
FLUSH_BYTES = 256 << 20


def step_flops(w) -> tuple[float, float]:
    f = 4.0 * w.B * w.H * w.Nq * w.Nk * w.d
    if w.causal:
        f /= 2
    return f, 2.5 * f


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def visible_pairs(w) -> int:
    """(query, key) pairs the mask leaves visible, per head."""
    if not w.causal:
        return w.Nq * w.Nk
    off = w.Nk - w.Nq if w.causal == "bottom_right" else 0
    return sum(max(0, min(w.Nk, q + off + 1)) for q in range(w.Nq))


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decoding forward: Q, K, V read once; O (16-bit) and LSE (fp32) written once."""
    return w.B * w.H * (2 * w.Nq * w.d * 2 + 2 * w.Nk * w.d * 2 + w.Nq * 4)


def config_dict(w, extra=None) -> dict:
    c = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
         "dtype": w.dtype, "sigma_qk": w.sigma_qk}
    if w.kind == "decode":
        c.update(kind="decode", bytes_per_step=decode_bytes(w), flops_per_step=4.0 * w.B * w.H * w.d * visible_pairs(w))
    elif w.kind == "kl":
        c.update(kind="kl", flops_per_step=sum(kl_flops(w)))
    else:
        c["flops_per_step"] = sum(step_flops(w))
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clocks and throttle reasons for one GPU."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        # samples go to a private temporary file (EXATTN_CLOCKS_CSV names another place to keep them)
        self.path = os.environ.get("EXATTN_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"exattn_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()

    def summary(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[5:9]))
            except Exception:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ oracle timing

def _oracle_step(x, w, n: int) -> float:
    """The oracle's forward + backward on head (0, 0) restricted to the first n queries and keys."""
    import oracle
    q = x["q"][:1, :1, :n]
    k = x["k"][:1, :1, :n]
    v = x["v"][:1, :1, :n]
    do = x["do"][:1, :1, :n]
    t = time.perf_counter()
    oracle.attn_fwd(q, k, v, w.causal, w.scale)
    oracle.attn_bwd(q, k, v, do, w.causal, w.scale)
    return time.perf_counter() - t


def _sample_flops(w, n: int) -> float:
    f = 4.0 * n * n * w.d * (0.5 if w.causal else 1.0)
    return 3.5 * f


def _pick_n(x, w, budget_s: float) -> int:
    import oracle
    oracle.build()
    n0 = min(256, w.Nq, w.Nk)
    t0 = max(_oracle_step(x, w, n0), 1e-4)
    n = int(n0 * math.sqrt(budget_s / t0))
    n = max(64, min(n, w.Nq, w.Nk))
    return n - n % 64 if n >= 128 else n


def cpu_baseline(x, w, budget_s: float = 15.0) -> dict:
    n = _pick_n(x, w, budget_s)
    dt = _oracle_step(x, w, n)
    return {"value": _sample_flops(w, n) / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 oracle forward+backward of head (b=0,h=0), first {n} queries and keys, "
                      f"{'causal' if w.causal else 'non-causal'}, d={w.d}; {dt:.1f} s on 1 thread "
                      f"(host has {len(os.sched_getaffinity(0))} cores available)",
            "seconds": dt}


def run_reference(args, w) -> None:
    from exact_head_attention_gb300 import workloads
    x = workloads.make_inputs(w)
    budget = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    n = _pick_n(x, w, budget)
    for _ in range(args.warmup):
        _oracle_step(x, w, n)
    times = [_oracle_step(x, w, n) for _ in range(args.steps)]
    med = statistics.median(times)
    value = _sample_flops(w, n) / med / 1e12
    sample = (f"per step: fp64 oracle forward+backward of head (b=0,h=0), first {n} queries and keys "
              f"(of {w.Nq}), 1 thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": med * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, {"sample_n": n}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ ranks

def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` over all ranks (identity when not distributed)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own batch (weak scaling), timed by the slowest rank."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def pipelined_e2e(steps: int, slots: list, h2d, compute, d2h, flush) -> tuple[float, float]:
    """End to end through the public API: pinned host inputs -> device -> one step -> pinned host results.

    Returns (ms per step with steps pipelined, ms of one step on its own).

    Pipelined: step i's host-to-device copies run on a copy-in stream, its kernels on a compute stream
    and its result copies on a copy-out stream.  Steps alternate between the device buffer sets in
    `slots`, so step i+1's inputs and step i-1's results cross the host link while step i computes.
    Events order the reuse of a set: its inputs are overwritten only after the compute that read them
    has finished, and its results only after the copy-out that read them has finished.  The time runs
    from the first copy-in to the last copy-out and includes filling and draining the pipeline.

    On its own: the same calls on one stream, one step at a time, each after an L2 flush (outside the
    events).  `h2d(slot)` and `d2h(slot)` issue copies on the current stream; `compute(slot, stream)`
    launches the step on `stream`."""
    import torch
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n_sl = len(slots)

    def run(n: int) -> float:
        cmp_done, out_done = [None] * n, [None] * n
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_in)
        for i in range(n):
            sl = slots[i % n_sl]
            if i >= n_sl:
                s_in.wait_event(cmp_done[i - n_sl])
            with torch.cuda.stream(s_in):
                h2d(sl)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
            s_cmp.wait_event(in_done)
            if i >= n_sl:
                s_cmp.wait_event(out_done[i - n_sl])
            compute(sl, s_cmp)
            cmp_done[i] = torch.cuda.Event()
            cmp_done[i].record(s_cmp)
            s_out.wait_event(cmp_done[i])
            with torch.cuda.stream(s_out):
                d2h(sl)
            out_done[i] = torch.cuda.Event()
            out_done[i].record(s_out)
        end.record(s_out)
        end.synchronize()
        return start.elapsed_time(end) / n

    run(3)
    pipe_ms = run(steps)
    alone = []
    for i in range(max(3, steps // 3)):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_cmp)
        with torch.cuda.stream(s_cmp):
            h2d(slots[0])
        compute(slots[0], s_cmp)
        with torch.cuda.stream(s_cmp):
            d2h(slots[0])
        b.record(s_cmp)
        b.synchronize()
        alone.append(a.elapsed_time(b))
    return pipe_ms, statistics.median(alone)


E2E_NOTE = ("pipelined over steps on three CUDA streams (copy-in, compute, copy-out) with two device buffer sets; "
            "the timed region runs from the first step's copy-in to the last step's copy-out, so filling and "
            "draining the pipeline are included; no L2 flush (each step's inputs arrive by host-to-device copy); "
            "alone_ms_per_step: one step by itself on one stream after an L2 flush")


# ------------------------------------------------------------------ main

def traffic_from_profile(kernel_key: str) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(path))[kernel_key]
    except Exception:
        return None
    if d.get("source_sha") != kernel_source_sha():
        return None
    return float(d["dram_bytes_per_launch"])


def kernel_source_sha() -> str:
    """Hash of what the headline kernels compile from, with comments and blank lines removed (a comment
    edit leaves the compiled kernels, and so the profiled traffic, unchanged): their translation units,
    the device headers they include (fwd_schedule.h: the persistent forward's argument; fwd_tile.cuh: the
    one-tile forward), and from
    kernels.h the argument structs they take and the integer constants (the other workloads' structs
    there do not change these kernels).  Host-only code is left out."""
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "attn_bwd.cu", "ptx.cuh", "kernels.h", "softmax.cuh", "kv_order.cuh", "fwd_schedule.h",
              "fwd_tile.cuh"):
        src = open(os.path.join(ROOT, "exact_head_attention_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        if f == "kernels.h":
            parts = [m.group(0) for m in re.finditer(r"struct (RowStrides|FwdArgs|BwdArgs) \{.*?\};", src, flags=re.S)]
            parts += re.findall(r"constexpr int [^;]*;", src)
            src = "\n".join(parts)
        h.update("\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ decoding workloads

DECODE_METRIC = "decoding attention forward (split-KV): algorithmic bytes per second"


def _oracle_decode_heads(x, w, nheads: int) -> float:
    import oracle
    t = time.perf_counter()
    for i in range(nheads):
        b, h = divmod(i, w.H)
        oracle.attn_fwd(x["q"][b:b + 1, h:h + 1], x["k"][b:b + 1, h:h + 1], x["v"][b:b + 1, h:h + 1], w.causal,
                        w.scale)
    return time.perf_counter() - t


def _decode_pick_heads(x, w, budget_s: float) -> int:
    import oracle
    oracle.build()
    t1 = max(_oracle_decode_heads(x, w, 1), 1e-4)
    return max(1, min(w.B * w.H, int(budget_s / t1)))


def decode_cpu_sample(x, w, nheads: int) -> tuple[float, float, str]:
    dt = _oracle_decode_heads(x, w, nheads)
    gbs = decode_bytes(w) * nheads / (w.B * w.H) / dt / 1e9
    sample = (f"fp64 oracle forward of the first {nheads} of {w.B * w.H} heads (all {w.Nq} queries, {w.Nk} keys), "
              f"{dt:.1f} s on 1 thread (host has {len(os.sched_getaffinity(0))} cores available)")
    return gbs, dt, sample


def run_decode(args, w, rank: int, world: int) -> None:
    from exact_head_attention_gb300 import workloads
    if args.impl == "reference":
        if rank != 0:
            return
        x = workloads.make_inputs(w, with_grad_out=False)
        nheads = _decode_pick_heads(x, w, max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup))))
        for _ in range(args.warmup):
            _oracle_decode_heads(x, w, nheads)
        times = [_oracle_decode_heads(x, w, nheads) for _ in range(args.steps)]
        med = statistics.median(times)
        value = decode_bytes(w) * nheads / (w.B * w.H) / med / 1e9
        sample = f"per step: fp64 oracle forward of the first {nheads} of {w.B * w.H} heads, 1 thread"
        print(json.dumps({
            "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": med * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, {"sample_heads": nheads}),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from exact_head_attention_gb300 import build as _build
    from exact_head_attention_gb300 import exattn
    _build.build()
    exattn.load()

    x = workloads.make_inputs(w, seed_offset=10 * rank, with_grad_out=False)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, _, sample = decode_cpu_sample(x, w, _decode_pick_heads(x, w, 15.0))
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample}

    stream = torch.cuda.current_stream()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    splits = exattn.splitkv_num_splits(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(max(256, exattn.splitkv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, splits)), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launch():
        st = exattn.fwd_splitkv_raw(q, k, v, o, lse, w.causal, w.scale, splits, ws)
        if st:
            raise RuntimeError(f"C-ABI status {st}: {exattn.last_error()}")

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}")
    for _ in range(args.warmup):
        launch()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        launch()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    ms_per_step = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in evs), dist, dev)

    # end to end: pinned host Q, K, V -> device -> split-KV forward -> host O, LSE
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse))

    slots = [{"q": q, "k": k, "v": v, "o": o, "lse": lse, "ws": ws}]
    slots.append({n: torch.empty_like(t) for n, t in slots[0].items()})

    def h2d_(sl):
        for n, ht in (("q", hq), ("k", hk), ("v", hv)):
            sl[n].copy_(ht, non_blocking=True)

    def compute_(sl, s):
        st = exattn.fwd_splitkv_raw(sl["q"], sl["k"], sl["v"], sl["o"], sl["lse"], w.causal, w.scale, splits, sl["ws"],
                                    stream=s)
        if st:
            raise RuntimeError(f"C-ABI status {st}: {exattn.last_error()}")

    def d2h_(sl):
        ho.copy_(sl["o"], non_blocking=True)
        hlse.copy_(sl["lse"], non_blocking=True)

    e2e_ms, alone_ms = pipelined_e2e(args.e2e_steps, slots, h2d_, compute_, d2h_, flush) if args.e2e_steps else (0, 0)
    sampler.stop()
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    alone_ms = max_over_ranks(alone_ms, dist, dev)

    nbytes = decode_bytes(w)
    pk = peaks()
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9  # the slice and merge kernels together
    line = {
        "metric": DECODE_METRIC, "value": world * nbytes / (ms_per_step * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp16", "data": "synthetic: seeded normal Q, K, V (sigma 1)",
        "config": config_dict(w, {"num_splits": splits, "parallelism": "replicas" if world > 1 else "single GPU",
                                  "l2": "256 MiB flush write between timed steps, outside the CUDA events"}),
        "fwd_tflops": 4.0 * w.B * w.H * w.d * visible_pairs(w) / (ms_per_step * 1e-3) / 1e12,
        "roofline": {"kernel": "fwd_split_kernel + fwd_combine_kernel (attn_fwd_splitkv)", "bound": "hbm",
                     "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": None, "peak_kind": f"HBM copy bandwidth ({pk['source']})"},
        "cpu_baseline": cpu,
        "e2e": ({"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "alone_ms_per_step": alone_ms,
                 "timing": E2E_NOTE} if args.e2e_steps else None),
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "wall_s_timed_region": t_wall1 - t_wall0,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ------------------------------------------------------------------ attention KL workloads

KL_METRIC = "attention KL divergence fwd+bwd TFLOPS (causal-adjusted; 2 forward + 4 backward score-sized products)"


def kl_flops(w) -> tuple[float, float]:
    one = 2.0 * w.B * w.H * w.Nq * w.Nk * w.d * (0.5 if w.causal else 1.0)  # one score-sized product
    return 2 * one, 4 * one


def _oracle_kl_step(x, w, n: int) -> float:
    import oracle
    sel = {k: v[:1, :1, :n] for k, v in x.items()}  # head (0, 0), first n rows (and keys)
    t = time.perf_counter()
    oracle.kl_fwd(sel["q1"], sel["k1"], sel["q2"], sel["k2"], w.causal, w.scale)
    oracle.kl_bwd(sel["q1"], sel["k1"], sel["q2"], sel["k2"], sel["g"], 1, w.causal, w.scale)
    return time.perf_counter() - t


def _kl_sample_flops(w, n: int) -> float:
    return 6.0 * 2.0 * n * n * w.d * (0.5 if w.causal else 1.0)


def _kl_pick_n(x, w, budget_s: float) -> int:
    import oracle
    oracle.build()
    n0 = min(256, w.Nq, w.Nk)
    t0 = max(_oracle_kl_step(x, w, n0), 1e-4)
    n = int(n0 * math.sqrt(budget_s / t0))
    n = max(64, min(n, w.Nq, w.Nk))
    return n - n % 64 if n >= 128 else n


def run_kl(args, w, rank: int, world: int) -> None:
    from exact_head_attention_gb300 import workloads
    if args.impl == "reference":
        if rank != 0:
            return
        x = workloads.make_kl_inputs(w)
        n = _kl_pick_n(x, w, max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup))))
        for _ in range(args.warmup):
            _oracle_kl_step(x, w, n)
        med = statistics.median(_oracle_kl_step(x, w, n) for _ in range(args.steps))
        value = _kl_sample_flops(w, n) / med / 1e12
        sample = f"per step: fp64 oracle KL forward + student backward of head (0,0), first {n} queries and keys, 1 thread"
        print(json.dumps({
            "impl": "reference", "metric": KL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": med * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, {"sample_n": n}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from exact_head_attention_gb300 import build as _build
    from exact_head_attention_gb300 import exattn
    _build.build()
    exattn.load()

    x = workloads.make_kl_inputs(w, seed_offset=10 * rank)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = _kl_pick_n(x, w, 15.0)
        dt = _oracle_kl_step(x, w, n)
        cpu = {"value": _kl_sample_flops(w, n) / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"fp64 oracle KL forward + student backward of head (0,0), first {n} queries and keys, "
                         f"{dt:.1f} s on 1 thread (host has {len(os.sched_getaffinity(0))} cores available)"}

    stream = torch.cuda.current_stream()
    d = {k: v.to(dev) for k, v in x.items()}
    kl, l1, l2 = (torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev) for _ in range(3))
    dq, dk = torch.empty_like(d["q2"]), torch.empty_like(d["k2"])
    kws = torch.empty(exattn.kl_bwd_workspace_size(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launch(ev=None):
        s1 = exattn.kl_fwd_raw(d["q1"], d["k1"], d["q2"], d["k2"], kl, l1, l2, w.causal, w.scale)
        if ev:
            ev[1].record(stream)
        s2 = exattn.kl_bwd_ex_raw(d["q1"], d["k1"], d["q2"], d["k2"], kl, l1, l2, d["g"], "student", dq, dk, w.causal,
                                  w.scale, args.kl_dq_mode, kws)
        if ev:
            ev[2].record(stream)
        if s1 or s2:
            raise RuntimeError(f"C-ABI status {(s1, s2)}: {exattn.last_error()}")

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}")
    for _ in range(args.warmup):
        launch()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        launch(evs[i])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    ms_per_step = max_over_ranks(fwd_ms + bwd_ms, dist, dev)

    # end to end: pinned host Q1, K1, Q2, K2, g -> device -> forward + backward -> host KL, dQ2, dK2
    h = {k: v.pin_memory() for k, v in x.items()}
    hkl = torch.empty(kl.shape, dtype=torch.float32).pin_memory()
    hdq, hdk = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk))
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in (hkl, hdq, hdk))

    slots = [dict(d, kl=kl, l1=l1, l2=l2, dq=dq, dk=dk, kws=kws)]
    slots.append({n: torch.empty_like(t) for n, t in slots[0].items()})

    def h2d_(sl):
        for k_ in d:
            sl[k_].copy_(h[k_], non_blocking=True)

    def compute_(sl, s):
        s1 = exattn.kl_fwd_raw(sl["q1"], sl["k1"], sl["q2"], sl["k2"], sl["kl"], sl["l1"], sl["l2"], w.causal, w.scale,
                               stream=s)
        s2 = exattn.kl_bwd_ex_raw(sl["q1"], sl["k1"], sl["q2"], sl["k2"], sl["kl"], sl["l1"], sl["l2"], sl["g"],
                                  "student", sl["dq"], sl["dk"], w.causal, w.scale, args.kl_dq_mode, sl["kws"], stream=s)
        if s1 or s2:
            raise RuntimeError(f"C-ABI status {(s1, s2)}: {exattn.last_error()}")

    def d2h_(sl):
        hkl.copy_(sl["kl"], non_blocking=True)
        hdq.copy_(sl["dq"], non_blocking=True)
        hdk.copy_(sl["dk"], non_blocking=True)

    e2e_ms, alone_ms = pipelined_e2e(args.e2e_steps, slots, h2d_, compute_, d2h_, flush) if args.e2e_steps else (0, 0)
    sampler.stop()
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    alone_ms = max_over_ranks(alone_ms, dist, dev)

    ff, bf = kl_flops(w)
    pk = peaks()
    achieved = bf / (bwd_ms * 1e-3) / 1e12
    line = {
        "metric": KL_METRIC, "value": world * (ff + bf) / (ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp16",
        "data": "synthetic: seeded normal teacher Q,K (sigma 1); student = teacher + noise (sigma %.2g); g ~ N(0,1)"
                % workloads.KL_STUDENT_NOISE,
        "config": config_dict(w, {"kind": "kl", "train": "student", "dq_mode": args.kl_dq_mode, "flops_per_step": ff + bf,
                                  "parallelism": "replicas" if world > 1 else "single GPU",
                                  "l2": "256 MiB flush write between timed steps, outside the CUDA events"}),
        "kernels_ms": {"kl_fwd": fwd_ms, "kl_bwd": bwd_ms},
        "fwd_tflops": ff / (fwd_ms * 1e-3) / 1e12, "bwd_tflops": achieved,
        "roofline": {"kernel": ("kl_bwd_fused_kernel with its pre and conversion launches (attn_kl_bwd_ex, one pass)"
                                if args.kl_dq_mode == "atomic" else "pair_dq_kernel + kl_dk_kernel (attn_kl_bwd)"),
                     "bound": "tensor", "achieved": achieved,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                     "traffic": None, "peak_kind": f"bf16 dense burst ({pk['source']})"},
        "cpu_baseline": cpu,
        "e2e": ({"value": world * (ff + bf) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                 "alone_ms_per_step": alone_ms, "timing": E2E_NOTE} if args.e2e_steps else None),
        # forward, then pre + one-pass kernel + dQ conversion (atomic) or the dQ and dK kernels
        "gpu_launches": (4 if args.kl_dq_mode == "atomic" else 3) * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "wall_s_timed_region": t_wall1 - t_wall0,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--dq-mode", choices=("atomic", "deterministic"), default="atomic",
                    help="attention workloads: dQ by reductions into the fp32 accumulator (attn_bwd) or by the "
                         "query-tile kernel (attn_bwd_ex, deterministic)")
    ap.add_argument("--kl-dq-mode", choices=("atomic", "deterministic"), default="atomic",
                    help="attention-KL workloads: the one-pass backward (atomic dQ) or the repeatable two-kernel one")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from exact_head_attention_gb300 import workloads
    w = workloads.WORKLOADS[args.workload or workloads.HEADLINE]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if w.kind == "decode":
        run_decode(args, w, rank, world)
        return
    if w.kind == "kl":
        run_kl(args, w, rank, world)
        return

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from exact_head_attention_gb300 import build as _build
    from exact_head_attention_gb300 import exattn
    _build.build()
    exattn.load()

    x = workloads.make_inputs(w, seed_offset=10 * rank)  # each rank: its own batch (tensor seeds use +0..3)
    cpu = cpu_baseline(x, w) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    stream = torch.cuda.current_stream()
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(exattn.workspace_size(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    deterministic = args.dq_mode == "deterministic"

    def backward_call(stream_=None):
        if deterministic:
            return exattn.bwd_ex_raw(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, "deterministic", ws, stream=stream_)
        return exattn.bwd_raw(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, ws, stream=stream_)

    def launch_step():
        """One step as a caller runs it: the forward, then the whole backward in one call."""
        st = (exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale), backward_call())
        if any(st):
            raise RuntimeError(f"C-ABI status {st}: {exattn.last_error()}")

    def launch(ev=None):
        """The same step with each backward launch called on its own and an event after every kernel (the
        deterministic mode: its whole backward between two events, reported as the key/value-block step)."""
        st = [exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale)]
        if ev:
            ev[1].record(stream)
        if deterministic:
            if ev:
                ev[2].record(stream)
            st.append(backward_call())
            if ev:
                ev[3].record(stream)
                ev[4].record(stream)
        else:
            for i, name in enumerate(exattn.BWD_STEPS):
                st.append(exattn.bwd_raw(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, ws, step=name))
                if ev:
                    ev[2 + i].record(stream)
        if any(st):
            raise RuntimeError(f"C-ABI status {st}: {exattn.last_error()}")

    for _ in range(args.warmup):
        launch_step()
        launch()
    torch.cuda.synchronize()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}")
    for _ in range(args.warmup):  # keep the GPU loaded while the sampler starts
        launch_step()
    # The timed region, two passes of K steps each.  Pass 1: whole steps, an event before and after each
    # (the backward's three launches are dependent launches that overlap one another's edges, which
    # events between them would prevent); it gives ms_per_step.  Pass 2: the same steps with an event
    # after every kernel; it gives the per-kernel times, and so the roofline's kernel duration.
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step_ev[i][0].record(stream)
        launch_step()
        step_ev[i][1].record(stream)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        launch(evs[i])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    if exattn.check_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms_per_step = max_over_ranks(statistics.median(step_ms), dist, dev)
    ms_per_step_mean = max_over_ranks(statistics.mean(step_ms), dist, dev)
    per = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)] for i in range(args.steps)]
    kern_names = ("fwd", "bwd_preprocess", "bwd_kv_blocks", "bwd_dq_convert")
    kern_ms = {name: statistics.median(p[j] for p in per) for j, name in enumerate(kern_names)}
    kern_ms_mean = {name: statistics.mean(p[j] for p in per) for j, name in enumerate(kern_names)}

    # end to end through the C ABI: pinned host inputs -> device -> fwd + bwd -> host outputs
    hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "do"))
    ho, hdq, hdk, hdv = (torch.empty_like(t, device="cpu").pin_memory() for t in (q, q, k, v))
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

    slots = [{"q": q, "k": k, "v": v, "do": do, "o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "ws": ws}]
    slots.append({n: torch.empty_like(t) for n, t in slots[0].items()})

    def h2d_(sl):
        for n, ht in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
            sl[n].copy_(ht, non_blocking=True)

    def compute_(sl, s):
        s1 = exattn.fwd_raw(sl["q"], sl["k"], sl["v"], sl["o"], sl["lse"], w.causal, w.scale, stream=s)
        s2 = exattn.bwd_ex_raw(sl["q"], sl["k"], sl["v"], sl["o"], sl["do"], sl["lse"], sl["dq"], sl["dk"], sl["dv"],
                               w.causal, w.scale, args.dq_mode, sl["ws"], stream=s)
        if s1 or s2:
            raise RuntimeError(exattn.last_error())

    def d2h_(sl):
        for ht, n in ((ho, "o"), (hlse, "lse"), (hdq, "dq"), (hdk, "dk"), (hdv, "dv")):
            ht.copy_(sl[n], non_blocking=True)

    e2e_ms, alone_ms = pipelined_e2e(args.e2e_steps, slots, h2d_, compute_, d2h_, flush) if args.e2e_steps else (0, 0)
    sampler.stop()
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    alone_ms = max_over_ranks(alone_ms, dist, dev)

    fwd_f, bwd_f = step_flops(w)
    flops = fwd_f + bwd_f
    value = job_throughput(flops, world, ms_per_step)
    pk = peaks()
    dominant = "bwd_kv_blocks"
    # the roofline's kernel duration is its mean over the timed launches (the step figures are medians)
    achieved = bwd_f / (kern_ms_mean[dominant] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp16",
        "data": "synthetic: seeded normal Q,K (sigma %.2g), V, dO (sigma 1)" % w.sigma_qk,
        "config": config_dict(w, {"parallelism": "replicas" if world > 1 else "single GPU",
                                  "l2": "256 MiB flush write between timed steps, outside the CUDA events",
                                  "dq_mode": args.dq_mode,
                                  "timing": "timed region = two passes of the steps: ms_per_step from CUDA "
                                            "events around each whole step (forward call, backward call); "
                                            "kernels_ms from the second pass, with an event after every kernel"}),
        "ms_per_step_mean": ms_per_step_mean,
        "pct_of_peak": 100.0 * (flops / (ms_per_step * 1e-3) / 1e12) / pk["bf16_tflops"],
        "peak_tflops": pk["bf16_tflops"], "peak_source": pk["source"],
        "pct_of_spec": 100.0 * (flops / (ms_per_step * 1e-3) / 1e12) / SPEC_BF16_TFLOPS,
        "spec_tflops": SPEC_BF16_TFLOPS,
        "kernels_ms": kern_ms, "kernels_ms_mean": kern_ms_mean,
        "fwd_tflops": fwd_f / (kern_ms["fwd"] * 1e-3) / 1e12,
        "bwd_tflops": bwd_f / (sum(kern_ms[n] for n in ("bwd_preprocess", "bwd_kv_blocks", "bwd_dq_convert")) * 1e-3) / 1e12,
        # each rate as a fraction of the measured bf16 tensor peak
        "frac_of_peak": {
            "fwd": fwd_f / (kern_ms["fwd"] * 1e-3) / 1e12 / pk["bf16_tflops"],
            "bwd": bwd_f / (sum(kern_ms[n] for n in ("bwd_preprocess", "bwd_kv_blocks", "bwd_dq_convert")) * 1e-3)
                   / 1e12 / pk["bf16_tflops"],
            "fwd_bwd": flops / (ms_per_step * 1e-3) / 1e12 / pk["bf16_tflops"],
        },
        "roofline": {"kernel": ("bwd_main_kernel + pair_dq_kernel (attn_bwd_ex, deterministic dQ)" if deterministic
                               else "bwd_main_kernel (attn_bwd_kv_blocks)"), "bound": "tensor", "achieved": achieved,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                     "traffic": None if deterministic else traffic_from_profile(f"{dominant}:{w.name}"),
                     "peak_kind": f"bf16 dense burst ({pk['source']})"},
        "cpu_baseline": ({k_: v_ for k_, v_ in cpu.items() if k_ != "seconds"} if cpu else None),
        "e2e": ({"value": job_throughput(flops, world, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "alone_ms_per_step": alone_ms,
                 "timing": E2E_NOTE} if args.e2e_steps else None),
        # both passes of the timed region: the forward, then preprocess + key/value blocks + conversion
        # (atomic) or preprocess + key/value blocks + query tiles (deterministic)
        "gpu_launches": 2 * 4 * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "wall_s_timed_region": t_wall1 - t_wall0,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
