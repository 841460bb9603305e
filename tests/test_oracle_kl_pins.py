"""Pins for the attention-KL oracle (no GPU).

The forward is pinned to library routines (scipy's softmax and relative
entropy on explicitly formed logits), to the attention oracle's LSE, and to
Gibbs' inequality, equality and a uniform-student closed form.  The two
backward settings are pinned to central finite differences of the oracle's own
forward and to torch autograd of the forward definition in fp64, plus the
zero-sum invariant of each dS row.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle


def _inputs(B, H, Nq, Nk, d, seed=0, spread=1.0):
    r = np.random.default_rng(seed)
    q1, k1, q2, k2 = (r.standard_normal(s) * spread for s in ((B, H, Nq, d), (B, H, Nk, d)) * 2)
    g = r.standard_normal((B, H, Nq))
    return q1, k1, q2, k2, g


def _allowed(causal, Nq, Nk):
    if not causal:
        return np.ones((Nq, Nk), bool)
    off = Nk - Nq if causal in (2, "bottom_right") else 0
    return np.tril(np.ones((Nq, Nk), bool), k=off)


@pytest.mark.parametrize("causal,Nq,Nk", [(0, 9, 13), (1, 12, 12), (2, 7, 15), (2, 15, 7)])
def test_kl_forward_matches_scipy(causal, Nq, Nk):
    q1, k1, q2, k2, _ = _inputs(2, 2, Nq, Nk, 8, seed=1)
    sc = 0.4
    kl, lse1, lse2 = oracle.kl_fwd(q1, k1, q2, k2, causal, sc)
    allowed = _allowed(causal, Nq, Nk)
    for b in range(2):
        for h in range(2):
            for q in range(Nq):
                vis = allowed[q]
                if not vis.any():
                    assert kl[b, h, q] == 0.0 and np.isneginf(lse1[b, h, q]) and np.isneginf(lse2[b, h, q])
                    continue
                s1 = sc * k1[b, h][vis] @ q1[b, h, q]
                s2 = sc * k2[b, h][vis] @ q2[b, h, q]
                p1, p2 = scipy.special.softmax(s1), scipy.special.softmax(s2)
                assert abs(kl[b, h, q] - scipy.special.rel_entr(p1, p2).sum()) < 1e-12
                assert abs(lse1[b, h, q] - scipy.special.logsumexp(s1)) < 1e-12
                assert abs(lse2[b, h, q] - scipy.special.logsumexp(s2)) < 1e-12


def test_kl_lse_equals_attention_lse():
    q1, k1, q2, k2, _ = _inputs(1, 3, 20, 30, 16, seed=2)
    _, lse1, lse2 = oracle.kl_fwd(q1, k1, q2, k2, 2, 0.25)
    v = np.zeros_like(k1)
    np.testing.assert_array_equal(lse1, oracle.attn_fwd(q1, k1, v, 2, 0.25)[1])
    np.testing.assert_array_equal(lse2, oracle.attn_fwd(q2, k2, v, 2, 0.25)[1])


def test_kl_gibbs_and_equality():
    q1, k1, q2, k2, _ = _inputs(2, 2, 16, 16, 8, seed=3, spread=2.0)
    kl, _, _ = oracle.kl_fwd(q1, k1, q2, k2, 1, 0.5)
    assert (kl >= -1e-15).all() and (kl > 1e-6).any()
    kl_same, l1, l2 = oracle.kl_fwd(q1, k1, q1, k1, 1, 0.5)
    assert (kl_same == 0.0).all()
    np.testing.assert_array_equal(l1, l2)


def test_kl_uniform_student_closed_form():
    """Q2 = 0: the student is uniform over the n visible keys, so KL = ln n - H(P1)."""
    q1, k1, _, k2, _ = _inputs(1, 1, 10, 10, 8, seed=4)
    q2 = np.zeros_like(q1)
    kl, _, lse2 = oracle.kl_fwd(q1, k1, q2, k2, 1, 0.7)
    n = np.arange(1, 11)
    np.testing.assert_allclose(lse2[0, 0], np.log(n), atol=1e-14)
    for q in range(10):
        p1 = scipy.special.softmax(0.7 * k1[0, 0, : q + 1] @ q1[0, 0, q])
        assert abs(kl[0, 0, q] - (math.log(q + 1) - scipy.special.entr(p1).sum())) < 1e-12


def _loss(q1, k1, q2, k2, g, causal, sc):
    kl, _, _ = oracle.kl_fwd(q1, k1, q2, k2, causal, sc)
    return float((g * kl).sum())


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal,Nq,Nk", [(0, 5, 6), (1, 6, 6), (2, 4, 7), (2, 7, 4)])
def test_kl_gradients_match_finite_differences(setting, causal, Nq, Nk):
    q1, k1, q2, k2, g = _inputs(1, 1, Nq, Nk, 4, seed=5)
    sc, h = 0.8, 1e-6
    dq, dk = oracle.kl_bwd(q1, k1, q2, k2, g, setting, causal, sc)
    names = ("q2", "k2") if setting == 1 else ("q1", "k1")
    for name, grad in zip(names, (dq, dk)):
        args = {"q1": q1, "k1": k1, "q2": q2, "k2": k2}
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args[name] = xp
            lp = _loss(args["q1"], args["k1"], args["q2"], args["k2"], g, causal, sc)
            args[name] = xm
            lm = _loss(args["q1"], args["k1"], args["q2"], args["k2"], g, causal, sc)
            num[idx] = (lp - lm) / (2 * h)
        args[name] = x
        err = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal,Nq,Nk", [(0, 33, 70), (1, 64, 64), (2, 40, 90)])
def test_kl_gradients_match_torch_autograd(setting, causal, Nq, Nk):
    B, H, d, sc = 2, 2, 16, 0.25
    q1, k1, q2, k2, g = _inputs(B, H, Nq, Nk, d, seed=6)
    t = {n: torch.from_numpy(a).requires_grad_(True) for n, a in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2))}
    allowed = torch.from_numpy(_allowed(causal, Nq, Nk))
    s1 = (sc * t["q1"] @ t["k1"].transpose(-1, -2)).masked_fill(~allowed, float("-inf"))
    s2 = (sc * t["q2"] @ t["k2"].transpose(-1, -2)).masked_fill(~allowed, float("-inf"))
    if setting == 1:
        s1 = s1.detach()
    else:
        s2 = s2.detach()
    zero = torch.zeros((), dtype=torch.float64)
    # masked entries are -inf; replace them by 0 before the product so that no 0 * inf reaches autograd
    lp1 = torch.where(allowed, torch.log_softmax(s1, -1), zero)
    lp2 = torch.where(allowed, torch.log_softmax(s2, -1), zero)
    terms = torch.where(allowed, lp1.exp() * (lp1 - lp2), zero)
    (torch.from_numpy(g) * terms.sum(-1)).sum().backward()
    dq, dk = oracle.kl_bwd(q1, k1, q2, k2, g, setting, causal, sc)
    tq, tk = (t["q2"], t["k2"]) if setting == 1 else (t["q1"], t["k1"])
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("setting", [1, 2])
def test_kl_gradient_invariants(setting):
    """Each dS row sums to 0, so sum_k dK_k = 0; identical distributions give zero gradients."""
    q1, k1, q2, k2, g = _inputs(2, 2, 24, 24, 8, seed=7)
    _, dk = oracle.kl_bwd(q1, k1, q2, k2, g, setting, 1, 0.5)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12 * max(1.0, np.abs(dk).max()) * 24
    dq0, dk0 = oracle.kl_bwd(q1, k1, q1, k1, g, setting, 1, 0.5)
    assert np.abs(dq0).max() < 1e-15 and np.abs(dk0).max() < 1e-15


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal,Nq,Nk", [(1, 40, 40), (2, 30, 50), (2, 50, 30)])
def test_kl_sampled_functions_match_full(setting, causal, Nq, Nk):
    B, H, d = 2, 2, 8
    q1, k1, q2, k2, g = _inputs(B, H, Nq, Nk, d, seed=8)
    kl, l1, l2 = oracle.kl_fwd(q1, k1, q2, k2, causal, 0.3)
    dq, dk = oracle.kl_bwd(q1, k1, q2, k2, g, setting, causal, 0.3)
    rows = np.array([0, 3, Nq - 1, Nq + 5, 3 * Nq + Nq - 1])
    bh, qi = rows // Nq, rows % Nq
    kl_r, l1_r, l2_r = oracle.kl_fwd_rows(q1, k1, q2, k2, causal, 0.3, rows)
    np.testing.assert_array_equal(kl_r, kl.reshape(-1, Nq)[bh, qi])
    np.testing.assert_array_equal(l1_r, l1.reshape(-1, Nq)[bh, qi])
    np.testing.assert_array_equal(l2_r, l2.reshape(-1, Nq)[bh, qi])
    np.testing.assert_allclose(oracle.kl_dq_rows(q1, k1, q2, k2, g, setting, causal, 0.3, rows),
                               dq.reshape(-1, Nq, d)[bh, qi], atol=1e-13)
    cols = np.array([0, 7, Nk - 1, Nk + 2, 2 * Nk + 11, 3 * Nk + Nk - 1])
    bk, ki = cols // Nk, cols % Nk
    np.testing.assert_allclose(oracle.kl_dk_cols(q1, k1, q2, k2, g, setting, causal, 0.3, cols),
                               dk.reshape(-1, Nk, d)[bk, ki], atol=1e-13)


@pytest.mark.parametrize("setting", [1, 2])
@pytest.mark.parametrize("causal,Nq,Nk", [(0, 21, 33), (1, 40, 40), (2, 50, 30)])
def test_kl_dk_column_parts_add_up_to_the_full_backward(setting, causal, Nq, Nk):
    """dK is a sum over query rows: the parts over a partition of [0, Nq) add up to oracle.kl_bwd's dK, and a
    part equals the full backward with g zeroed outside its rows (dK is linear in g)."""
    B, H, d = 2, 2, 8
    q1, k1, q2, k2, g = _inputs(B, H, Nq, Nk, d, seed=9)
    _, dk = oracle.kl_bwd(q1, k1, q2, k2, g, setting, causal, 0.3)
    cols = np.array([0, 1, Nk // 2, Nk - 1, Nk + 2, 3 * Nk + Nk - 1])
    bk, ki = cols // Nk, cols % Nk
    edges = [0, 3, 3, Nq // 2, Nq]
    parts = [oracle.kl_dk_cols(q1, k1, q2, k2, g, setting, causal, 0.3, cols, q_range=(a, b))
             for a, b in zip(edges[:-1], edges[1:])]
    np.testing.assert_allclose(sum(parts), dk.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
    g_part = np.zeros_like(g)
    g_part[:, :, 3:Nq // 2] = g[:, :, 3:Nq // 2]
    _, dk_p = oracle.kl_bwd(q1, k1, q2, k2, g_part, setting, causal, 0.3)
    np.testing.assert_allclose(parts[2], dk_p.reshape(-1, Nk, d)[bk, ki], atol=1e-13)
