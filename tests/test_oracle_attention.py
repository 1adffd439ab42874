"""Pins for the C fp64 attention oracle (oracle/attn_oracle.c).

Each test checks the oracle against something other than itself: the worked
example the pages print, brute force in pure Python loops, a float64 library
special case (torch CPU softmax/matmul), closed forms, invariances, central
finite differences of the forward, and identities of the softmax Jacobian.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_worked_examples.json")


def rnd(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


# ---------------------------------------------------------------- worked example

def test_worked_example_through_attention():
    """Scores 7, 4, 3 (then 9) realised as q.k with V = identity: row 0 of O is
    the weight vector and LSE is max + ln(denominator), as printed in
    carrie-l.github.io 上篇 section 四."""
    with open(GOLDEN) as f:
        ex = [e for e in json.load(f)["examples"] if e["id"] == "scores_7_4_3_then_9"][0]
    N = d = 4
    q = np.zeros((1, 1, N, d))
    q[0, 0, :, 0] = 1.0
    k = np.zeros((1, 1, N, d))
    k[0, 0, :, 0] = ex["scores_first"] + [ex["score_added"]]
    v = np.eye(N)[None, None]
    tol = ex["tol"]
    o, lse = oracle.attention_fwd(q, k, v, 1.0, kv_len=[3])          # only 7, 4, 3 visible
    np.testing.assert_allclose(o[0, 0, 0, :3], ex["weights_first"], atol=tol)
    assert o[0, 0, 0, 3] == 0.0
    assert abs(math.exp(lse[0, 0, 0] - 7) - ex["denominator_first"]) <= tol
    o, lse = oracle.attention_fwd(q, k, v, 1.0)                      # 9 added
    assert abs(math.exp(lse[0, 0, 0] - 9) - ex["denominator_after"]) <= tol
    np.testing.assert_allclose(o[0, 0, 0] * ex["denominator_after"], ex["exp_shifted_after"],
                               atol=2 * tol)


# ---------------------------------------------------------------- brute force

def brute_force(q, k, v, scale, causal, kv_len):
    B, H, N, d = q.shape
    O = np.zeros_like(q)
    L = np.zeros((B, H, N))
    for b in range(B):
        ln = N if kv_len is None else kv_len[b]
        for h in range(H):
            for i in range(N):
                vis = [j for j in range(N) if j < ln and not (causal and j > i)]
                s = {j: scale * sum(q[b, h, i, t] * k[b, h, j, t] for t in range(d)) for j in vis}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in vis)
                for t in range(d):
                    O[b, h, i, t] = sum(math.exp(s[j] - m) / z * v[b, h, j, t] for j in vis)
                L[b, h, i] = m + math.log(z)
    return O, L


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [3, 5]), (True, [2, 4])])
def test_brute_force_loops(causal, kv):
    rng = np.random.default_rng(10)
    q, k, v = (rnd(rng, 2, 2, 5, 3, s=1.5) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.6, causal=causal, kv_len=kv)
    O, L = brute_force(q, k, v, 0.6, causal, kv)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- library special case

@pytest.mark.parametrize("N,d,causal,pad", [(64, 16, False, False), (64, 16, True, False),
                                            (48, 8, False, True), (37, 32, True, True)])
def test_torch_float64_library(N, d, causal, pad):
    rng = np.random.default_rng(N + d)
    B, H = 2, 3
    q, k, v = (rnd(rng, B, H, N, d, s=2.0) for _ in range(3))
    kv = [N - 5, N // 2] if pad else None
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=causal, kv_len=kv)
    tq, tk, tv = (torch.from_numpy(t) for t in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    mask = torch.zeros(B, 1, N, N, dtype=torch.bool)
    if causal:
        mask |= torch.ones(N, N, dtype=torch.bool).triu(1)
    if pad:
        for b in range(B):
            mask[b, :, :, kv[b]:] = True
    s = s.masked_fill(mask, float("-inf"))
    np.testing.assert_allclose(o, (torch.softmax(s, -1) @ tv).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_v():
    rng = np.random.default_rng(11)
    q, k, v = (rnd(rng, 2, 2, 1, 7) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.3, causal=True)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.3 * (q * k).sum(-1), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [9, 20])])
def test_identical_keys_give_mean_of_visible_values(causal, kv):
    rng = np.random.default_rng(12)
    B, H, N, d = 2, 2, 20, 6
    q, v = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    k = np.broadcast_to(rnd(rng, B, H, 1, d), (B, H, N, d)).copy()
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal=causal, kv_len=kv)
    for b in range(B):
        ln = N if kv is None else kv[b]
        for i in range(N):
            n = min(i + 1, ln) if causal else ln
            np.testing.assert_allclose(o[b, :, i], v[b, :, :n].mean(axis=1), atol=1e-12)
            np.testing.assert_allclose(lse[b, :, i], 0.5 * (q[b, :, i] * k[b, :, 0]).sum(-1)
                                       + math.log(n), atol=1e-12)


def test_dominant_score_selects_its_value_row():
    rng = np.random.default_rng(13)
    N, d = 16, 4
    q = np.zeros((1, 1, N, d))
    q[..., 0] = 1.0
    k = rnd(rng, 1, 1, N, d, s=0.1)
    star = 11
    k[0, 0, star, 0] = 80.0                     # score gap > 70: other weights < e^-70
    v = rnd(rng, 1, 1, N, d)
    o, _ = oracle.attention_fwd(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, star], (N, d)), atol=1e-25 + 1e-15)


# ---------------------------------------------------------------- invariances

def test_key_shift_and_value_shift():
    rng = np.random.default_rng(14)
    B, H, N, d = 1, 2, 24, 5
    q, k, v = (rnd(rng, B, H, N, d) for _ in range(3))
    c = rnd(rng, d)
    o, lse = oracle.attention_fwd(q, k, v, 0.8, causal=True)
    o2, lse2 = oracle.attention_fwd(q, k + c, v, 0.8, causal=True)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse + 0.8 * (q @ c), atol=1e-12)
    o3, lse3 = oracle.attention_fwd(q, k, v + c, 0.8, causal=True)
    np.testing.assert_allclose(o3, o + c, atol=1e-12)
    np.testing.assert_allclose(lse3, lse, atol=0)


def test_key_permutation_noncausal():
    rng = np.random.default_rng(15)
    B, H, N, d = 2, 1, 30, 4
    q, k, v = (rnd(rng, B, H, N, d) for _ in range(3))
    perm = rng.permutation(N)
    o, lse = oracle.attention_fwd(q, k, v, 1.1)
    o2, lse2 = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], 1.1)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


def test_rows_entry_matches_full_forward():
    rng = np.random.default_rng(16)
    N, d = 40, 8
    q, k, v = (rnd(rng, 1, 1, N, d) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.4, causal=True, kv_len=[33])
    rows = [0, 5, 32, 33, 39]
    orow, lrow = oracle.attention_fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.4, causal=True,
                                           kv_len=33)
    np.testing.assert_array_equal(orow, o[0, 0, rows])
    np.testing.assert_array_equal(lrow, lse[0, 0, rows])


def test_recompute_p_from_lse():
    """P_ij = exp(S_ij - L_i) rebuilds O from the saved statistic alone
    (magicnetworld section 八; llm-training-tutorial 4.3.4)."""
    rng = np.random.default_rng(17)
    N, d = 33, 6
    q, k, v = (rnd(rng, 1, 1, N, d, s=2) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.9, causal=True)
    S = 0.9 * q[0, 0] @ k[0, 0].T
    S[np.triu_indices(N, 1)] = -np.inf
    P = np.exp(S - lse[0, 0][:, None])
    np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-13)
    np.testing.assert_allclose(P @ v[0, 0], o[0, 0], atol=1e-12)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, scale, causal, kv):
    o, _ = oracle.attention_fwd(q, k, v, scale, causal=causal, kv_len=kv, threads=1)
    return float((o * do).sum())


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [5, 9]), (True, [7, 4])])
def test_backward_central_finite_differences(causal, kv):
    rng = np.random.default_rng(20)
    B, H, N, d = 2, 1, 9, 4
    q, k, v, do = (rnd(rng, B, H, N, d) for _ in range(4))
    scale = 0.7
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, scale, causal, kv)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, scale, causal, kv)
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-30)
        assert err <= 1e-6, (name, err)


def test_backward_identities():
    rng = np.random.default_rng(21)
    B, H, N, d = 2, 2, 31, 8
    q, k, v, do = (rnd(rng, B, H, N, d, s=1.5) for _ in range(4))
    kv = [31, 17]
    dq, dk, dv, D = oracle.attention_bwd(q, k, v, do, 0.5, causal=True, kv_len=kv)
    o, _ = oracle.attention_fwd(q, k, v, 0.5, causal=True, kv_len=kv)
    # D two ways: sum_j P_ij dP_ij == rowsum(dO o O)
    np.testing.assert_allclose(D, (do * o).sum(-1), atol=1e-12)
    # softmax rows of dS sum to zero, so the key gradients of each head sum to zero
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12 * np.abs(dk).max() * N)
    # padded keys get exactly zero gradient
    assert np.all(dk[1, :, 17:] == 0.0) and np.all(dv[1, :, 17:] == 0.0)


def test_backward_uniform_attention_closed_form():
    """Identical keys make P uniform over the visible keys: then dQ = 0 and
    dV_j = sum over queries i that see j of dO_i / n_i."""
    rng = np.random.default_rng(22)
    B, H, N, d = 1, 2, 12, 5
    q, v, do = (rnd(rng, B, H, N, d) for _ in range(3))
    k = np.broadcast_to(rnd(rng, B, H, 1, d), (B, H, N, d)).copy()
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, do, 0.9, causal=True)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    ref = np.zeros_like(dv)
    for j in range(N):
        for i in range(j, N):
            ref[:, :, j] += do[:, :, i] / (i + 1)
    np.testing.assert_allclose(dv, ref, atol=1e-13)
