"""Pins for the oracle's attention variants: grouped K/V heads (GQA / MQA)
and flash-attn's (left, right) sliding window.

Each test checks the oracle against something other than itself: brute force
in pure Python loops, a float64 library special case (torch CPU softmax with
an explicit mask), closed forms (a window of one key, identical keys), the
reduction of grouped heads to multi-head attention with repeated K/V, and
central finite differences of the forward.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rnd(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


def visible(i, j, causal, ln, wl, wr):
    return (j < ln and not (causal and j > i) and not (wl >= 0 and j < i - wl)
            and not (wr >= 0 and j > i + wr))


def brute_force(q, k, v, scale, causal, kv_len, wl, wr):
    """Pure-Python loops; K/V head of query head h is h // (H // H_kv)."""
    B, H, N, d = q.shape
    G = H // k.shape[1]
    O = np.zeros_like(q)
    L = np.zeros((B, H, N))
    for b in range(B):
        ln = N if kv_len is None else kv_len[b]
        for h in range(H):
            hk = h // G
            for i in range(N):
                vis = [j for j in range(N) if visible(i, j, causal, ln, wl, wr)]
                if not vis:
                    L[b, h, i] = -math.inf
                    continue
                s = {j: scale * sum(q[b, h, i, t] * k[b, hk, j, t] for t in range(d)) for j in vis}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in vis)
                for t in range(d):
                    O[b, h, i, t] = sum(math.exp(s[j] - m) / z * v[b, hk, j, t] for j in vis)
                L[b, h, i] = m + math.log(z)
    return O, L


@pytest.mark.parametrize("Hkv,causal,kv,win", [
    (2, False, None, (1, 2)), (1, True, None, (3, -1)), (2, False, [4, 7], (2, 0)),
    (1, False, [3, 7], (0, 3)), (4, True, [6, 2], (1, 1)), (2, False, None, (-1, 1)),
])
def test_brute_force_loops(Hkv, causal, kv, win):
    rng = np.random.default_rng(30)
    B, H, N, d = 2, 4, 7, 3
    q = rnd(rng, B, H, N, d, s=1.5)
    k, v = rnd(rng, B, Hkv, N, d, s=1.5), rnd(rng, B, Hkv, N, d, s=1.5)
    o, lse = oracle.attention_fwd(q, k, v, 0.6, causal=causal, kv_len=kv, window=win)
    O, L = brute_force(q, k, v, 0.6, causal, kv, *win)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    fin = np.isfinite(L)
    np.testing.assert_allclose(lse[fin], L[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("N,d,causal,win", [(64, 16, False, (5, 7)), (64, 16, True, (9, -1)),
                                            (48, 8, False, (0, 20)), (37, 32, True, (12, 0))])
def test_torch_float64_library(N, d, causal, win):
    rng = np.random.default_rng(N + d + 1)
    B, H = 2, 3
    q, k, v = (rnd(rng, B, H, N, d, s=2.0) for _ in range(3))
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal=causal, window=win)
    tq, tk, tv = (torch.from_numpy(t) for t in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    mask = torch.zeros(N, N, dtype=torch.bool)
    if causal:
        mask |= j > i
    if win[0] >= 0:
        mask |= j < i - win[0]
    if win[1] >= 0:
        mask |= j > i + win[1]
    s = s.masked_fill(mask, float("-inf"))
    np.testing.assert_allclose(o, (torch.softmax(s, -1) @ tv).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_window_of_one_key_gives_its_value():
    rng = np.random.default_rng(31)
    q, k, v = (rnd(rng, 2, 2, 9, 5) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.4, window=(0, 0))
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.4 * (q * k).sum(-1), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal,kv,win", [(False, None, (3, 2)), (True, None, (4, -1)),
                                           (False, [9, 20], (2, 5)), (True, [6, 20], (1, 0)),
                                           (False, [5, 20], (0, -1))])
def test_identical_keys_mean_over_window(causal, kv, win):
    """With every key equal, P is uniform over the visible keys: O_i is the
    mean of V over [max(0, i-left), min(len-1, i+right)] (right = 0 under
    causal) and LSE_i = scale q_i.k + ln(count); empty windows give O = 0 and
    LSE = -inf."""
    rng = np.random.default_rng(32)
    B, H, N, d = 2, 2, 20, 6
    q, v = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    k = np.broadcast_to(rnd(rng, B, H, 1, d), (B, H, N, d)).copy()
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal=causal, kv_len=kv, window=win)
    wl, wr = win
    for b in range(B):
        ln = N if kv is None else kv[b]
        for i in range(N):
            lo = 0 if wl < 0 else max(0, i - wl)
            hi = ln - 1 if wr < 0 else min(ln - 1, i + wr)
            if causal:
                hi = min(hi, i)
            n = hi - lo + 1
            if n <= 0:
                assert np.all(o[b, :, i] == 0.0) and np.all(np.isneginf(lse[b, :, i]))
                continue
            np.testing.assert_allclose(o[b, :, i], v[b, :, lo:hi + 1].mean(axis=1), atol=1e-12)
            np.testing.assert_allclose(lse[b, :, i], 0.5 * (q[b, :, i] * k[b, :, 0]).sum(-1)
                                       + math.log(n), atol=1e-12)


def test_window_wider_than_sequence_is_no_window():
    rng = np.random.default_rng(33)
    q, k, v = (rnd(rng, 1, 2, 13, 4) for _ in range(3))
    a = oracle.attention_fwd(q, k, v, 0.7, causal=True)
    b = oracle.attention_fwd(q, k, v, 0.7, causal=True, window=(13, 13))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal,win", [(False, (-1, -1)), (True, (3, -1)), (False, (2, 4))])
def test_grouped_heads_equal_repeated_kv(causal, win):
    """GQA with H_kv heads equals multi-head attention whose K/V heads are the
    grouped ones repeated H / H_kv times; dK, dV of a group are the sums of
    the repeated heads' gradients."""
    rng = np.random.default_rng(34)
    B, H, Hkv, N, d = 2, 6, 2, 11, 4
    G = H // Hkv
    q, do = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    k, v = rnd(rng, B, Hkv, N, d), rnd(rng, B, Hkv, N, d)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    kv = [11, 8]
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal=causal, kv_len=kv, window=win)
    o2, lse2 = oracle.attention_fwd(q, kr, vr, 0.5, causal=causal, kv_len=kv, window=win)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    dq, dk, dv, D = oracle.attention_bwd(q, k, v, do, 0.5, causal=causal, kv_len=kv, window=win)
    dq2, dk2, dv2, D2 = oracle.attention_bwd(q, kr, vr, do, 0.5, causal=causal, kv_len=kv,
                                             window=win)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(D, D2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, G, N, d).sum(2), atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, G, N, d).sum(2), atol=1e-12)


@pytest.mark.parametrize("Hkv,causal,kv,win", [(1, False, None, (2, 1)), (2, True, [7, 4], (3, -1)),
                                                (1, True, None, (1, 0))])
def test_backward_central_finite_differences(Hkv, causal, kv, win):
    rng = np.random.default_rng(35)
    B, H, N, d = 2, 2, 7, 3
    q, do = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    k, v = rnd(rng, B, Hkv, N, d), rnd(rng, B, Hkv, N, d)
    scale = 0.7
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv, window=win)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal=causal, kv_len=kv, threads=1,
                                    window=win)
        return float((o * do).sum())

    h = 1e-6
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
        err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-30)
        assert err <= 1e-6, (name, err)


def test_rejects_bad_groupings():
    rng = np.random.default_rng(36)
    q = rnd(rng, 1, 4, 5, 2)
    k = rnd(rng, 1, 3, 5, 2)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, k, 1.0)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, q, q, 1.0, window=(-2, 0))
