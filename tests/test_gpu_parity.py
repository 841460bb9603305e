"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Small and ragged shapes are compared element by element over every output.
The standard, encoder-decoder and long-sequence (8k) workloads are compared
element by element over every head (one oracle call per head on a thread
pool), and the two very-long-context (32k) workloads over their first and
last heads (query rows split over threads).  Every head of the long workloads
is also checked at full size on sampled query rows (O, LSE, dQ) and key rows
(dK, dV) that the oracle evaluates one by one -- the last key rows and the
rows of the first key blocks, which every query tile adds into under a
causal mask -- plus gradient invariants that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_head_attention_gb300 import workloads

from parity import (check_fwd, check_grads, f64_head, heavy_cols, oracle_cols_threaded, oracle_every_head,
                    oracle_heads, oracle_one_head_split, rel_l2, run_gpu, sample_rows)

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS

# (B, H, Nq, Nk, d, dtype, causal): one tile, several tiles, ragged tails, Nq != Nk both ways, degenerate sizes
SMALL = [
    (1, 2, 128, 128, 64, "fp16", False),
    (1, 2, 128, 128, 64, "fp16", True),
    (1, 1, 1, 1, 64, "bf16", False),
    (1, 1, 1, 1, 128, "bf16", True),
    (1, 1, 7, 7, 64, "bf16", True),
    (1, 2, 100, 100, 128, "bf16", True),
    (2, 1, 129, 257, 64, "bf16", False),
    (1, 1, 257, 129, 128, "fp16", True),
    (1, 1, 257, 129, 64, "bf16", False),
    (1, 2, 1000, 1000, 64, "bf16", True),
    (1, 1, 300, 700, 128, "bf16", False),
    (1, 1, 700, 300, 64, "fp16", True),
    (1, 1, 513, 513, 128, "bf16", True),
    (3, 2, 384, 384, 128, "fp16", False),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}q{}k{}d{}{}{}".format(*s[:6], "c" if s[6] else ""))
def test_small_full_parity(shape):
    B, H, Nq, Nk, d, dt, causal = shape
    w = workloads.custom(B, H, Nq, Nk, d, dt, causal)
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
    check_fwd(w, got["o"], got["lse"], o, lse, w.name)
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, w.name)


@pytest.mark.parametrize("name", ["tiny_fp16"])
def test_tiny_workload_full(name):
    w = W[name]
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    check_fwd(w, got["o"], got["lse"], o, lse, name)
    dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale)
    check_grads(got, {"dq": dq, "dk": dk, "dv": dv}, name)


@pytest.mark.parametrize("name", ["self1k_bf16", "self1k_causal_bf16", "dec_self512_fp16", "dec_cross512x1024_fp16"])
def test_midsize_workloads_every_head(name):
    """The standard self-attention and encoder-decoder workloads in full: every output of every head against
    the oracle (one oracle call per head, on a thread pool)."""
    w = W[name]
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    ref = oracle_every_head(w, x)
    check_fwd(w, got["o"], got["lse"], ref["o"], ref["lse"], name)
    check_grads(got, ref, name)
    _check_invariants(w, x, got, name)


def test_long_sequence_workload_every_element():
    """The long-sequence workload (B=1, H=12, N=8192, d=128, causal, sigma 1.5) in full: every element of O,
    LSE, dQ, dK and dV of all twelve heads against the oracle (one oracle call per head, on a thread pool),
    in the launch configuration the benchmark times."""
    w = W["long8k_causal_bf16"]
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    ref = oracle_every_head(w, x)
    check_fwd(w, got["o"], got["lse"], ref["o"], ref["lse"], w.name)
    errs = check_grads(got, ref, w.name)
    # per head as well: a head whose gradients were wrong could hide in the 12-head norm
    for h in range(w.H):
        check_grads({k: got[k][0, h] for k in ("dq", "dk", "dv")}, {k: ref[k][0, h] for k in ("dq", "dk", "dv")},
                    f"{w.name} head {h}")
    assert max(errs.values()) <= 2e-2


@pytest.mark.parametrize("name", ["ctx32k_d128_causal_bf16", "ctx32k_d64_causal_bf16"])
def test_very_long_context_two_heads_every_element(name):
    """The very-long-context workloads (B=1, H=8, N=32768, causal, d=128 and d=64): every element of the first
    and the last head against the oracle, its query rows split over a thread pool; the other heads are
    checked on sampled rows and key rows and through invariants (test_long_workloads_full_size_sampled)."""
    w = W[name]
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        ref = oracle_one_head_split(w, x, b, h)
        check_fwd(w, got["o"][b, h], got["lse"][b, h], ref["o"], ref["lse"], f"{name} head ({b},{h})")
        check_grads({k: got[k][b, h] for k in ("dq", "dk", "dv")}, ref, f"{name} head ({b},{h})")


def _check_invariants(w, x, got, what):
    """Per head: sum_k dK_k = 0 (rows of dS sum to 0) and sum_k dV_k = sum_q dO_q (rows of P sum to 1).

    Both hold at any size; the bound is relative to the head's ||dK||_F and ||sum_q dO_q||."""
    dk = got["dk"].astype(np.float64)
    dk_sum = np.linalg.norm(dk.sum(axis=2), axis=-1)
    dk_norm = np.linalg.norm(dk, axis=(2, 3))
    assert (dk_sum <= 2e-2 * dk_norm + 1e-6).all(), f"{what}: sum_k dK_k != 0 ({(dk_sum / dk_norm).max():.2e})"
    dv_sum = got["dv"].astype(np.float64).sum(axis=2)
    do_sum = x["do"].double().sum(dim=2).numpy()
    err = np.linalg.norm(dv_sum - do_sum, axis=-1) / np.maximum(np.linalg.norm(do_sum, axis=-1), 1e-30)
    assert (err <= 2e-2).all(), f"{what}: sum_k dV_k != sum_q dO_q ({err.max():.2e})"


def _heavy_cols_check(w, x, got, b, h):
    """dK and dV of head (b, h) on the rows of its first key blocks and one in the middle.  Under a causal mask
    the first keys are seen by every query row, so these rows accumulate over all query tiles (the key block
    that does the most work); the oracle evaluates every query row for them, split over threads."""
    cols = heavy_cols(w.Nk)
    xs = {n: f64_head(x[n], b, h) for n in ("q", "k", "v", "do")}

    def part(r):
        return oracle.attn_dkdv_cols(xs["q"], xs["k"], xs["v"], xs["do"], w.causal, w.scale, cols, q_range=r)

    dk_c, dv_c = oracle_cols_threaded(part, w.Nq, w.Nk, w.causal)
    check_grads({"dk": got["dk"][b, h, cols], "dv": got["dv"][b, h, cols]}, {"dk": dk_c, "dv": dv_c},
                f"{w.name} head ({b},{h}) dK/dV rows {cols.tolist()}")


def _sampled_check(w, x, got, n_rows, heads, seed, heavy=True):
    N = w.Nq
    for (b, h) in heads:
        if heavy:
            _heavy_cols_check(w, x, got, b, h)
        bh = b * w.H + h
        rows = sample_rows(N, n_rows, seed + bh)
        flat = bh * N + rows
        o_r, lse_r = oracle.attn_fwd_rows(x["q"], x["k"], x["v"], w.causal, w.scale, flat)
        check_fwd(w, got["o"][b, h, rows], got["lse"][b, h, rows], o_r, lse_r, f"{w.name} head {bh}")
        dq_r, _ = oracle.attn_dq_rows(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, flat)
        check_grads({"dq": got["dq"][b, h, rows]}, {"dq": dq_r}, f"{w.name} head {bh} dQ rows")
        # key rows near the end: few query rows see them under the causal mask, so the oracle is cheap
        cols = np.array(sorted({w.Nk - 1, w.Nk - 2, w.Nk - 64, w.Nk - 129, w.Nk - 200}), dtype=np.int64)
        dk_c, dv_c = oracle.attn_dkdv_cols(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, bh * w.Nk + cols)
        check_grads({"dk": got["dk"][b, h, cols], "dv": got["dv"][b, h, cols]}, {"dk": dk_c, "dv": dv_c},
                    f"{w.name} head {bh} dK/dV rows")


@pytest.mark.parametrize("name", ["long8k_causal_bf16", "ctx32k_d64_causal_bf16", "ctx32k_d128_causal_bf16"])
def test_long_workloads_full_size_sampled(name):
    w = W[name]
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    _sampled_check(w, x, got, 48 if w.Nq > 10000 else 96, heads, seed=w.index)
    _check_invariants(w, x, got, name)


def test_many_heads_causal_accumulator_beyond_l2_sampled():
    """64 heads of 8192 causal rows: a 256 MiB dQ accumulator, twice the L2, so the key blocks are launched
    in groups of a few heads instead of heads fastest (the last group taking the remainder); sampled rows
    against the oracle."""
    w = workloads.custom(4, 16, 8192, 8192, 128, "bf16", True, index=32)
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    for (b, h) in [(0, 0), (1, 7), (3, 15)]:
        # the oracle sees one head at a time, so its row indices are the head's own
        xs = {n: x[n][b:b + 1, h:h + 1] for n in ("q", "k", "v", "do")}
        gs = {n: got[n][b:b + 1, h:h + 1] for n in ("o", "lse", "dq", "dk", "dv")}
        ws = workloads.custom(1, 1, w.Nq, w.Nk, w.d, "bf16", True, index=32)
        _sampled_check(ws, xs, gs, 32, [(0, 0)], seed=w.index + b * w.H + h)
    _check_invariants(w, x, got, w.name)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "nomask"])
def test_more_heads_than_a_grid_y_dimension(causal):
    """B*H = 66000 heads of 8 rows: more than the 65535 a grid's y dimension allows, so the key/value
    blocks' one-dimensional numbering (and its head groups: the 2 GiB accumulator is far past L2) is what
    reaches every head; the first, a middle and the last heads against the oracle, every head finite."""
    w = workloads.custom(1100, 60, 8, 8, 64, "bf16", causal, index=34)
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    heads = [(0, 0), (550, 31), (1099, 59)]
    ref = oracle_heads(w, x, heads)
    sel = lambda a: np.stack([a[b, h] for b, h in heads])  # noqa: E731
    check_fwd(w, sel(got["o"]), sel(got["lse"]), ref["o"], ref["lse"], w.name)
    check_grads({k: sel(got[k]) for k in ("dq", "dk", "dv")}, ref, w.name)
    for k in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[k]).all(), k


@pytest.mark.parametrize("shape", [(1, 1, 200003, 200003, 64, "bf16", True),
                                   (1, 1, 100001, 131075, 128, "bf16", "bottom_right")],
                         ids=["q200003_d64_causal", "q100001_k131075_d128_bottom_right"])
def test_very_long_sequences_sampled(shape):
    """Sequences far past the workloads' 32k: tensor-map row coordinates above 2^17, ~1500 key blocks,
    a ragged last tile; sampled rows and the last key rows against the oracle."""
    w = workloads.custom(*shape, index=31)
    x = workloads.make_inputs(w)
    got = run_gpu(w, x)
    # the first key rows here would need every one of 100k-200k query rows evaluated in full: the tail only
    _sampled_check(w, x, got, 24, [(0, 0)], seed=w.index, heavy=False)


def test_outputs_written_everywhere():
    """Outputs pre-filled with NaN must be fully overwritten (ragged shapes included)."""
    from exact_head_attention_gb300 import exattn
    w = workloads.custom(2, 3, 333, 271, 128, "bf16", True)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.Nq), float("nan"), device=dev)
    assert exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale) == 0
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ws = torch.full((exattn.workspace_size(w.B, w.H, w.Nq, w.d),), 0xFF, dtype=torch.uint8, device=dev)
    assert exattn.bwd_raw(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, ws) == 0
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("shape", [(1, 12, 8192, 8192, 128, "bf16", True), (1, 12, 8192, 8192, 64, "fp16", True)],
                         ids=["8k_causal_d128", "8k_causal_d64"])
def test_every_query_block_written_by_the_packed_forward(shape):
    """Causal shapes whose forward runs one CTA per SM over host-packed lists of query blocks (12 heads of
    32 blocks: too coarse for an even spread over the SMs in launch order): O and LSE pre-filled with NaN
    must be overwritten everywhere (every block is on exactly one list), and a second call must give the
    same bits."""
    from exact_head_attention_gb300 import exattn
    w = workloads.custom(*shape, index=35)
    _require_packed(w)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.H, w.Nq), float("nan"), device=dev)
        assert exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale) == 0
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    for o, lse in outs:
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def _require_packed(w):
    """Skip unless this device runs the shape's forward from packed lists (the plan depends on the SM count)."""
    from exact_head_attention_gb300 import exattn
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lists = exattn.fwd_schedule(w.B, w.H, w.Nq, w.Nk, w.d, w.causal, sm_count=sms)
    if lists is None:
        pytest.skip(f"the forward of this shape runs in launch order on {sms} SMs")
    return lists


def test_packed_forward_bottom_right_ragged_sampled():
    """A list-scheduled causal forward with the bottom-right mask and a ragged last block (Nq = 8000,
    Nk = 9000): sampled rows of three heads, the last rows included, against the oracle."""
    w = workloads.custom(1, 12, 8000, 9000, 128, "bf16", "bottom_right", index=36)
    _require_packed(w)
    x = workloads.make_inputs(w)
    got = run_gpu(w, x, backward=False)
    for h in (0, 5, 11):
        xs = {n: x[n][:, h:h + 1] for n in ("q", "k", "v")}
        rows = np.array(sorted(set(sample_rows(w.Nq, 40, 36 + h).tolist()) | {7999, 7998, 7936, 7935}), dtype=np.int64)
        o_r, lse_r = oracle.attn_fwd_rows(xs["q"], xs["k"], xs["v"], w.causal, w.scale, rows)
        check_fwd(w, got["o"][0, h, rows], got["lse"][0, h, rows], o_r, lse_r, f"{w.name} head {h}")


def test_packed_forward_blocks_without_keys():
    """Bottom-right mask with more queries than keys (Nq = 9000, Nk = 8000): rows q < 1000 see no key, so the
    first three 256-row blocks of every head have no key tile, and the packed lists put them behind blocks
    that do.  Such a block skips the loads and products and writes O = 0, LSE = -inf; the block after it on
    the same list must still run normally.  O and LSE are pre-filled with NaN; every head's key-less rows
    are checked exactly and sampled rows (the boundary at q = 1000 included) against the oracle."""
    from exact_head_attention_gb300 import exattn
    w = workloads.custom(1, 12, 9000, 8000, 128, "bf16", "bottom_right", index=37)
    lists = _require_packed(w)
    nqb = -(-w.Nq // 256)
    assert any(any(b % nqb < 3 for b in lst[1:]) for lst in lists), "no key-less block follows another block"
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.Nq), float("nan"), device=dev)
    assert exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale) == 0
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert (o[:, :, :1000] == 0).all() and np.isneginf(lse[:, :, :1000]).all()
    assert np.isfinite(o).all() and np.isfinite(lse[:, :, 1000:]).all()
    for h in (0, 6, 11):
        xs = {n: x[n][:, h:h + 1] for n in ("q", "k", "v")}
        rows = np.array(sorted(set(sample_rows(w.Nq, 32, 37 + h).tolist()) | {998, 999, 1000, 1001, 1023, 1024}),
                        dtype=np.int64)
        o_r, lse_r = oracle.attn_fwd_rows(xs["q"], xs["k"], xs["v"], w.causal, w.scale, rows)
        check_fwd(w, o[0, h, rows], lse[0, h, rows], o_r, lse_r, f"{w.name} head {h}")


@pytest.mark.parametrize("shape", [(2, 3, 700, 300, 64, "fp16", "bottom_right"), (1, 2, 1500, 2048, 64, "bf16", True),
                                   (3, 1, 257, 129, 64, "bf16", "bottom_right")],
                         ids=["nq700_nk300_bottom_right", "nq1500_nk2048", "nq257_nk129_bottom_right"])
def test_one_tile_forward_every_output(shape):
    """The causal forward at d = 64 over at most 2048 keys runs one query tile per CTA, two CTAs per SM:
    every output against the oracle, with O and LSE pre-filled with NaN.  With the bottom-right mask and
    more queries than keys, whole query tiles see no key (their CTAs load nothing and write O = 0,
    LSE = -inf) while the CTA beside them on the SM runs a normal tile."""
    from exact_head_attention_gb300 import exattn
    w = workloads.custom(*shape, index=38)
    assert exattn.fwd_schedule(w.B, w.H, w.Nq, w.Nk, w.d, w.causal, sm_count=152) is None
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.Nq), float("nan"), device=dev)
    assert exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale) == 0
    torch.cuda.synchronize()
    assert exattn.check_device_error() == 0
    ref_o, ref_lse = oracle.attn_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    check_fwd(w, o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, w.name)


def test_guard_bytes_untouched():
    """Writes stay inside the outputs: sentinel bytes around each output are unchanged."""
    from exact_head_attention_gb300 import exattn
    w = workloads.custom(1, 2, 200, 150, 64, "fp16", False)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    pad = 4096

    def guarded(like):
        n = like.numel()
        buf = torch.full((n + 2 * pad,), 12345.0, dtype=like.dtype, device=dev)
        return buf, buf[pad:pad + n].view(like.shape)

    ob, o = guarded(q)
    lb, lse = guarded(torch.empty((w.B, w.H, w.Nq), dtype=torch.float32))
    assert exattn.fwd_raw(q, k, v, o, lse, w.causal, w.scale) == 0
    qb, dq = guarded(q)
    kb, dk = guarded(k)
    vb, dv = guarded(v)
    ws = torch.empty(exattn.workspace_size(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)
    assert exattn.bwd_raw(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, ws) == 0
    torch.cuda.synchronize()
    for buf in (ob, lb, qb, kb, vb):
        assert (buf[:pad] == 12345.0).all() and (buf[-pad:] == 12345.0).all()


def test_repeatable_forward_and_dkdv():
    """Forward and dK/dV are bitwise repeatable; dQ (fp32 atomics) agrees within rounding."""
    w = workloads.custom(1, 4, 1024, 1024, 128, "bf16", True)
    x = workloads.make_inputs(w)
    a = run_gpu(w, x)
    b = run_gpu(w, x)
    for key in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[key], b[key]), key
    assert rel_l2(a["dq"], b["dq"]) < 1e-3
