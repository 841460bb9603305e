"""Pins for the CPU oracle (no GPU): each check fixes the oracle to something
other than itself -- closed forms, invariants, hand-derived worked examples,
central finite differences, and the special case that reduces to a library
routine (torch's fp64 CPU scaled_dot_product_attention with autograd).

A plausible slip in the oracle (a dropped scale, a transposed operand, a wrong
mask direction, a missing D term, a sign) fails at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, sigma=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * sigma


def _qkv(B, H, Nq, Nk, d, seed=0, sigma=1.0):
    return (_rand((B, H, Nq, d), seed, sigma), _rand((B, H, Nk, d), seed + 1, sigma),
            _rand((B, H, Nk, d), seed + 2), _rand((B, H, Nq, d), seed + 3))


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(7, 7), (5, 9), (9, 5)])
def test_probability_rows_sum_to_one(causal, Nq, Nk):
    q, k, _, _ = _qkv(1, 1, Nq, Nk, 6, seed=1)
    p, lse = oracle.attn_probs(q[0, 0], k[0, 0], causal, 0.4)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert (p >= 0).all()
    if causal:  # top-left mask: nothing above the diagonal
        for qi in range(Nq):
            assert (p[qi, qi + 1:] == 0).all()
            assert (p[qi, : min(qi + 1, Nk)] > 0).all()
    # LSE is the log of the normaliser of the scaled scores (checked via torch.logsumexp)
    s = 0.4 * q[0, 0] @ k[0, 0].T
    if causal:
        s = np.where(np.tril(np.ones((Nq, Nk), dtype=bool)), s, -np.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(s), dim=1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_v(causal):
    q, k, _, _ = _qkv(2, 3, 11, 11, 8, seed=2)
    vrow = _rand((8,), 99)
    v = np.broadcast_to(vrow, (2, 3, 11, 8)).copy()
    o, _ = oracle.attn_fwd(q, k, v, causal, 0.35)
    np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), atol=1e-13)


def test_causal_row_zero_is_v0():
    q, k, v, _ = _qkv(2, 2, 9, 9, 5, seed=3)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.7)
    np.testing.assert_allclose(o[:, :, 0, :], v[:, :, 0, :], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.7 * np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0]), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_closed_form(causal):
    """Q = 0 makes every visible score 0: P is uniform over the visible keys."""
    B, H, N, d = 1, 2, 10, 4
    _, k, v, do = _qkv(B, H, N, N, d, seed=4)
    q = np.zeros((B, H, N, d))
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.5)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, 0.5)
    if not causal:
        np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
        np.testing.assert_allclose(lse, math.log(N), atol=1e-13)
        np.testing.assert_allclose(dv, np.broadcast_to(do.sum(axis=2, keepdims=True) / N, dv.shape), atol=1e-13)
        # dQ_q = scale/N * sum_k (dO_q . (V_k - Vbar)) K_k
        vc = v - v.mean(axis=2, keepdims=True)
        ref = 0.5 / N * np.einsum("bhqc,bhkc,bhke->bhqe", do, vc, k)
        np.testing.assert_allclose(dq, ref, atol=1e-13)
    else:
        cnt = np.arange(1, N + 1)[:, None]
        np.testing.assert_allclose(o, np.cumsum(v, axis=2) / cnt, atol=1e-13)
        np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), atol=1e-13)
        # dV_k = sum_{q >= k} dO_q / (q + 1)
        w = do / cnt
        ref = np.flip(np.cumsum(np.flip(w, axis=2), axis=2), axis=2)
        np.testing.assert_allclose(dv, ref, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)  # dK = scale dS^T Q with Q = 0


def test_single_key():
    q, k, v, do = _qkv(1, 2, 6, 1, 3, seed=5)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.9)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :, :1, :], o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, 0.9 * np.einsum("bhqc,bhc->bhq", q, k[:, :, 0]), atol=1e-13)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, False, 0.9)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv[:, :, 0], do.sum(axis=2), atol=1e-13)


def test_one_hot_permutation():
    """Orthonormal query rows and K = lambda * Q[perm]: P is (nearly) a permutation matrix."""
    N = d = 8
    rng = np.random.default_rng(6)
    qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    perm = rng.permutation(N)
    q = qm[None, None]
    k = 80.0 * qm[perm][None, None]
    v = _rand((1, 1, N, d), 7)
    o, _ = oracle.attn_fwd(q, k, v, False, 1.0)
    inv = np.argsort(perm)  # query i matches key inv[i]
    np.testing.assert_allclose(o[0, 0], v[0, 0, inv], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums(causal):
    """sum_k dK_k = 0 (dS rows sum to 0) and sum_k dV_k = sum_q dO_q (P rows sum to 1)."""
    q, k, v, do = _qkv(2, 2, 12, 12, 5, seed=8)
    _, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, 0.45)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_D_equals_rowsum_dO_O(causal):
    q, k, v, do = _qkv(1, 2, 9, 9, 4, seed=9)
    o, _ = oracle.attn_fwd(q, k, v, causal, 0.6)
    _, _, _, D = oracle.attn_bwd(q, k, v, do, causal, 0.6)
    np.testing.assert_allclose(D, (do * o).sum(axis=-1), atol=1e-12)


# ---------------------------------------------------------- worked examples

def _ev(x):
    if isinstance(x, list):
        return [_ev(e) for e in x]
    return float(eval(x, {"__builtins__": {}}, {"log": math.log}))


def test_hand_worked_examples():
    cases = json.load(open(os.path.join(GOLDEN, "hand_worked_2x2.json")))["cases"]
    for c in cases:
        arr = {key: np.array(_ev(c[key]))[None] for key in ("Q", "K", "V", "dO", "O", "dQ", "dK", "dV")}
        lse_ref = np.array(_ev(c["LSE"]))[None]
        sc = _ev(c["scale"])
        o, lse = oracle.attn_fwd(arr["Q"], arr["K"], arr["V"], c["causal"], sc)
        np.testing.assert_allclose(o, arr["O"], atol=1e-13, err_msg=c["name"])
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13, err_msg=c["name"])
        dq, dk, dv, _ = oracle.attn_bwd(arr["Q"], arr["K"], arr["V"], arr["dO"], c["causal"], sc)
        np.testing.assert_allclose(dq, arr["dQ"], atol=1e-13, err_msg=c["name"])
        np.testing.assert_allclose(dk, arr["dK"], atol=1e-13, err_msg=c["name"])
        np.testing.assert_allclose(dv, arr["dV"], atol=1e-13, err_msg=c["name"])


# ------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal,Nq,Nk", [(False, 8, 8), (True, 8, 8), (False, 5, 7), (True, 7, 5)])
def test_gradients_match_finite_differences(causal, Nq, Nk):
    d, sc, h = 4, 0.8, 1e-6
    q, k, v, do = _qkv(1, 1, Nq, Nk, d, seed=10)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, sc)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, causal, sc)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


# ------------------------------------------- library special case (torch SDPA)

@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 128, 128, 64), False),
    ((1, 2, 128, 128, 64), True),
    ((2, 3, 33, 70, 16), False),
    ((2, 3, 70, 33, 16), True),
    ((1, 1, 1, 1, 8), False),
])
def test_matches_torch_fp64_sdpa(shape, causal):
    B, H, Nq, Nk, d = shape
    q, k, v, do = _qkv(B, H, Nq, Nk, d, seed=11)
    sc = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc)
    to.backward(torch.from_numpy(do))
    o, lse = oracle.attn_fwd(q, k, v, causal, sc)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, sc)
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
    s = sc * torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2)
    if causal:
        s = s.masked_fill(~torch.ones(Nq, Nk, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


# ------------------------------------------ sampled functions == full ones

@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_and_cols_match_full(causal):
    B, H, Nq, Nk, d = 2, 2, 40, 40, 8
    q, k, v, do = _qkv(B, H, Nq, Nk, d, seed=12)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.3)
    dq, dk, dv, D = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    rows = np.array([0, 5, 39, 40 + 7, 3 * 40 + 39])
    bh, qi = rows // Nq, rows % Nq
    o_r, lse_r = oracle.attn_fwd_rows(q, k, v, causal, 0.3, rows)
    np.testing.assert_allclose(o_r, o.reshape(-1, Nq, d)[bh, qi], atol=1e-13)
    np.testing.assert_allclose(lse_r, lse.reshape(-1, Nq)[bh, qi], atol=1e-13)
    dq_r, D_r = oracle.attn_dq_rows(q, k, v, do, causal, 0.3, rows)
    np.testing.assert_allclose(dq_r, dq.reshape(-1, Nq, d)[bh, qi], atol=1e-13)
    np.testing.assert_allclose(D_r, D.reshape(-1, Nq)[bh, qi], atol=1e-13)
    cols = np.array([0, 17, 39, 40 + 1, 2 * 40 + 20, 3 * 40 + 39])
    bk, ki = cols // Nk, cols % Nk
    dk_c, dv_c = oracle.attn_dkdv_cols(q, k, v, do, causal, 0.3, cols)
    np.testing.assert_allclose(dk_c, dk.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    np.testing.assert_allclose(dv_c, dv.reshape(-1, Nk, d)[bk, ki], atol=1e-13)


# ------------------------------------------------- bottom-right causal mask

def test_bottom_right_square_is_top_left():
    q, k, v, do = _qkv(1, 2, 24, 24, 8, seed=20)
    for f in (lambda c: oracle.attn_fwd(q, k, v, c, 0.4), lambda c: oracle.attn_bwd(q, k, v, do, c, 0.4)):
        for a, b in zip(f(1), f(2)):
            np.testing.assert_array_equal(a, b)


def test_bottom_right_single_query_sees_every_key():
    q, k, v, do = _qkv(2, 1, 1, 37, 8, seed=21)
    for a, b in zip(oracle.attn_bwd(q, k, v, do, 0, 0.4), oracle.attn_bwd(q, k, v, do, "bottom_right", 0.4)):
        np.testing.assert_array_equal(a, b)
    o0, l0 = oracle.attn_fwd(q, k, v, False, 0.4)
    o2, l2 = oracle.attn_fwd(q, k, v, 2, 0.4)
    np.testing.assert_array_equal(o0, o2)
    np.testing.assert_array_equal(l0, l2)


@pytest.mark.parametrize("Nq", [1, 9, 30])
def test_bottom_right_is_suffix_of_square_causal(Nq):
    """The last Nq queries of a square top-left problem, posed alone with bottom-right alignment,
    give the same rows of O, LSE, dQ; with dO zero on the leading rows, the same dK, dV."""
    Nk, d = 30, 8
    qf, k, v, dof = _qkv(1, 2, Nk, Nk, d, seed=22)
    dof[:, :, : Nk - Nq] = 0.0
    qs, dos = qf[:, :, Nk - Nq:], dof[:, :, Nk - Nq:]
    of, lf = oracle.attn_fwd(qf, k, v, True, 0.35)
    os_, ls = oracle.attn_fwd(qs, k, v, "bottom_right", 0.35)
    np.testing.assert_array_equal(os_, of[:, :, Nk - Nq:])
    np.testing.assert_array_equal(ls, lf[:, :, Nk - Nq:])
    dqf, dkf, dvf, _ = oracle.attn_bwd(qf, k, v, dof, True, 0.35)
    dqs, dks, dvs, _ = oracle.attn_bwd(qs, k, v, dos, "bottom_right", 0.35)
    np.testing.assert_array_equal(dqs, dqf[:, :, Nk - Nq:])
    np.testing.assert_allclose(dks, dkf, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dvs, dvf, rtol=0, atol=1e-15)


@pytest.mark.parametrize("Nq,Nk", [(20, 45), (45, 20), (64, 64)])
def test_bottom_right_matches_torch_masked_sdpa(Nq, Nk):
    B, H, d = 1, 2, 16
    q, k, v, do = _qkv(B, H, Nq, Nk, d, seed=23)
    sc = 1.0 / math.sqrt(d)
    allowed = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    seen = allowed.any(dim=1).numpy()  # rows that see at least one key
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq[:, :, seen], tk, tv, attn_mask=allowed[torch.from_numpy(seen)], scale=sc)
    to.backward(torch.from_numpy(do[:, :, seen]))
    o, lse = oracle.attn_fwd(q, k, v, 2, sc)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, 2, sc)
    np.testing.assert_allclose(o[:, :, seen], to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq[:, :, seen], tq.grad.numpy()[:, :, seen], atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
    # rows that see no key: zero output, -inf LSE, zero dQ
    assert np.all(o[:, :, ~seen] == 0.0) and np.all(dq[:, :, ~seen] == 0.0)
    assert np.all(np.isneginf(lse[:, :, ~seen]))
    s = sc * torch.from_numpy(q[:, :, seen]) @ torch.from_numpy(k).transpose(-1, -2)
    s = s.masked_fill(~allowed[torch.from_numpy(seen)], float("-inf"))
    np.testing.assert_allclose(lse[:, :, seen], torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


@pytest.mark.parametrize("Nq,Nk", [(5, 7), (7, 5)])
def test_bottom_right_gradients_match_finite_differences(Nq, Nk):
    d, sc, h = 4, 0.8, 1e-6
    q, k, v, do = _qkv(1, 1, Nq, Nk, d, seed=24)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, 2, sc)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, 2, sc)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = {"q": q, "k": k, "v": v}
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("Nq,Nk", [(30, 40), (40, 30)])
def test_bottom_right_sampled_rows_and_cols_match_full(Nq, Nk):
    B, H, d = 2, 2, 8
    q, k, v, do = _qkv(B, H, Nq, Nk, d, seed=25)
    o, lse = oracle.attn_fwd(q, k, v, 2, 0.3)
    dq, dk, dv, D = oracle.attn_bwd(q, k, v, do, 2, 0.3)
    rows = np.array([0, 5, Nq - 1, Nq + 7, 3 * Nq + Nq - 1])
    bh, qi = rows // Nq, rows % Nq
    o_r, lse_r = oracle.attn_fwd_rows(q, k, v, 2, 0.3, rows)
    np.testing.assert_allclose(o_r, o.reshape(-1, Nq, d)[bh, qi], atol=1e-13)
    np.testing.assert_array_equal(lse_r, lse.reshape(-1, Nq)[bh, qi])
    dq_r, D_r = oracle.attn_dq_rows(q, k, v, do, 2, 0.3, rows)
    np.testing.assert_allclose(dq_r, dq.reshape(-1, Nq, d)[bh, qi], atol=1e-13)
    cols = np.array([0, 17, Nk - 1, Nk + 1, 2 * Nk + 20, 3 * Nk + Nk - 1])
    bk, ki = cols // Nk, cols % Nk
    dk_c, dv_c = oracle.attn_dkdv_cols(q, k, v, do, 2, 0.3, cols)
    np.testing.assert_allclose(dk_c, dk.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    np.testing.assert_allclose(dv_c, dv.reshape(-1, Nk, d)[bk, ki], atol=1e-13)


# ------------------------------- query-row parts of the column-sampled gradients

@pytest.mark.parametrize("causal,Nq,Nk", [(0, 37, 29), (1, 40, 40), (2, 30, 50), (2, 50, 30)])
def test_dkdv_column_parts_add_up_to_the_full_backward(causal, Nq, Nk):
    """dK_k and dV_k are sums over query rows: the parts over the rows of a partition of [0, Nq) (empty parts,
    parts without visible keys included) add up to oracle_attn_bwd's full gradients, and a part equals the
    full backward of the same rows with dO zeroed elsewhere."""
    B, H, d = 2, 2, 8
    q, k, v, do = _qkv(B, H, Nq, Nk, d, seed=31)
    _, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    cols = np.array([0, 1, Nk // 2, Nk - 1, Nk + 3, 3 * Nk + Nk - 1])
    bk, ki = cols // Nk, cols % Nk
    edges = [0, 0, 5, 6, Nq // 2, Nq - 1, Nq]
    parts = [oracle.attn_dkdv_cols(q, k, v, do, causal, 0.3, cols, q_range=(a, b))
             for a, b in zip(edges[:-1], edges[1:])]
    np.testing.assert_allclose(sum(p[0] for p in parts), dk.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    np.testing.assert_allclose(sum(p[1] for p in parts), dv.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    # rows [6, Nq/2) alone (parts[3]): dK and dV are linear in dO given P (D too), so zeroing dO outside the
    # rows gives the same part
    do_part = np.zeros_like(do)
    do_part[:, :, 6:Nq // 2] = do[:, :, 6:Nq // 2]
    _, dk_p, dv_p, _ = oracle.attn_bwd(q, k, v, do_part, causal, 0.3)
    np.testing.assert_allclose(parts[3][0], dk_p.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    np.testing.assert_allclose(parts[3][1], dv_p.reshape(-1, Nk, d)[bk, ki], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_threaded_heavy_columns_equal_the_serial_oracle(causal):
    """The GPU tests' threaded evaluation of the first key rows (parts over query rows on a thread pool,
    summed) equals one serial oracle call."""
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from parity import heavy_cols, oracle_cols_threaded, query_parts

    Nq, Nk, d = 700, 900, 16
    q, k, v, do = _qkv(1, 1, Nq, Nk, d, seed=32)
    mask = {False: 0, True: 1, "bottom_right": 2}[causal]
    cols = heavy_cols(Nk)
    want = oracle.attn_dkdv_cols(q, k, v, do, mask, 0.25, cols)
    got = oracle_cols_threaded(lambda r: oracle.attn_dkdv_cols(q, k, v, do, mask, 0.25, cols, q_range=r),
                               Nq, Nk, causal, workers=5)
    for a, b in zip(got, want):
        np.testing.assert_allclose(a, b, atol=1e-12)
    parts = query_parts(Nq, Nk, causal, 5)
    assert parts[0][0] == 0 and parts[-1][1] == Nq and all(a < b for a, b in parts)
    assert all(parts[i][1] == parts[i + 1][0] for i in range(len(parts) - 1))


def test_threaded_whole_head_helpers_equal_the_plain_oracle():
    """The GPU tests' whole-head oracle runs -- one oracle call per head on a thread pool, and one long head
    split into query-row parts -- equal the plain single-call oracle (rows without keys included)."""
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from exact_head_attention_gb300 import workloads
    from parity import oracle_every_head, oracle_one_head_split

    for causal in (False, True, "bottom_right"):
        w = workloads.custom(2, 3, 300, 260, 32, "bf16", causal)
        x = workloads.make_inputs(w)
        o, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, w.scale)
        dq, dk, dv, _ = oracle.attn_bwd(x["q"], x["k"], x["v"], x["do"], causal, w.scale)
        ref = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
        every = oracle_every_head(w, x, workers=3)
        one = oracle_one_head_split(w, x, 1, 2, workers=5)
        for key, want in ref.items():
            np.testing.assert_array_equal(every[key], want)
            np.testing.assert_allclose(one[key], want[1, 2], atol=1e-12)
