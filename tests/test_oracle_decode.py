"""Pins for the oracle's decode-shaped attention (Nq queries at the end of a
Nk-key cache): it reduces to the pinned square forward when Nq = Nk, to a
float64 library softmax for one query, and matches pure-Python brute force
with padding and windows, including queries that see no key."""
import math

import numpy as np
import pytest
import torch

import oracle


def rnd(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("causal,win", [(False, None), (True, None), (True, (5, -1))])
def test_square_case_is_the_forward(causal, win):
    rng = np.random.default_rng(40)
    q = rnd(rng, 2, 4, 23, 8)
    k, v = rnd(rng, 2, 2, 23, 8), rnd(rng, 2, 2, 23, 8)
    o, lse = oracle.attention_decode(q, k, v, 0.4, causal=causal, window=win)
    o2, lse2 = oracle.attention_fwd(q, k, v, 0.4, causal=causal, window=win)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_one_query_is_a_library_softmax():
    rng = np.random.default_rng(41)
    B, H, Nk, d = 2, 3, 57, 16
    q, k, v = rnd(rng, B, H, 1, d), rnd(rng, B, H, Nk, d), rnd(rng, B, H, Nk, d)
    kv = [57, 31]
    o, lse = oracle.attention_decode(q, k, v, 0.25, causal=True, kv_len=kv)
    for b in range(B):
        n = kv[b]
        s = 0.25 * torch.from_numpy(q[b]) @ torch.from_numpy(k[b, :, :n]).transpose(-1, -2)
        np.testing.assert_allclose(o[b], (torch.softmax(s, -1) @ torch.from_numpy(v[b, :, :n])).numpy(),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def brute(q, k, v, scale, causal, kv_len, win):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    G = H // k.shape[1]
    wl, wr = (-1, -1) if win is None else win
    O, L = np.zeros_like(q), np.zeros((B, H, Nq))
    for b in range(B):
        ln = Nk if kv_len is None else kv_len[b]
        for h in range(H):
            for t in range(Nq):
                pos = ln - Nq + t
                vis = [j for j in range(Nk) if j < ln and not (causal and j > pos)
                       and not (wl >= 0 and j < pos - wl) and not (wr >= 0 and j > pos + wr)]
                if not vis:
                    L[b, h, t] = -math.inf
                    continue
                s = {j: scale * sum(q[b, h, t, c] * k[b, h // G, j, c] for c in range(d)) for j in vis}
                m = max(s.values())
                z = sum(math.exp(x - m) for x in s.values())
                for c in range(d):
                    O[b, h, t, c] = sum(math.exp(s[j] - m) / z * v[b, h // G, j, c] for j in vis)
                L[b, h, t] = m + math.log(z)
    return O, L


@pytest.mark.parametrize("causal,kv,win", [(True, [11, 2], None), (False, [7, 11], (3, 1)),
                                           (True, None, (2, -1))])
def test_brute_force(causal, kv, win):
    rng = np.random.default_rng(42)
    q = rnd(rng, 2, 4, 3, 3)
    k, v = rnd(rng, 2, 2, 11, 3), rnd(rng, 2, 2, 11, 3)
    o, lse = oracle.attention_decode(q, k, v, 0.7, causal=causal, kv_len=kv, window=win)
    O, L = brute(q, k, v, 0.7, causal, kv, win)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    fin = np.isfinite(L)
    np.testing.assert_allclose(lse[fin], L[fin], rtol=0, atol=1e-13)
