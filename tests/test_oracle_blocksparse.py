"""Pins for the oracle's block mask (Block-Sparse FlashAttention: a coarse
block-level mask matrix whose zero entries hide whole (query block, key
block) pairs, "炉案与百步之外的仓库…" 第八部分).

Each test checks the oracle against something other than itself:
- brute force in pure Python loops with the mask expanded element by element;
- central finite differences of the forward, for the backward;
- a block-diagonal mask, which splits attention into independent
  sub-sequences computed without a mask;
- a lower-triangular block mask, which under the causal mask changes nothing.
Plausible mistakes (a transposed mask, the wrong block size or row length, a
mask applied to queries instead of keys) fail at least one of them.
"""
import math

import numpy as np
import pytest

import oracle


def rnd(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


def brute_force(q, k, v, scale, causal, kv_len, bm, bs):
    B, H, N, d = q.shape
    G = H // k.shape[1]
    O = np.zeros_like(q)
    L = np.zeros((B, H, N))
    for b in range(B):
        ln = N if kv_len is None else kv_len[b]
        for h in range(H):
            hk = h // G
            for i in range(N):
                vis = [j for j in range(N)
                       if j < ln and not (causal and j > i) and bm[i // bs][j // bs]]
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


@pytest.mark.parametrize("bs,causal,kv,Hkv", [(3, False, None, 2), (3, True, None, 1),
                                              (4, False, [5, 10], 2), (2, True, [9, 3], 1)])
def test_brute_force_loops(bs, causal, kv, Hkv):
    rng = np.random.default_rng(60 + bs)
    B, H, N, d = 2, 2, 10, 3            # N not a multiple of bs: a ragged last block
    q = rnd(rng, B, H, N, d, s=1.5)
    k, v = rnd(rng, B, Hkv, N, d, s=1.5), rnd(rng, B, Hkv, N, d, s=1.5)
    t = -(-N // bs)
    bm = (rng.random((t, t)) < 0.55).astype(np.uint8)
    bm[0, t - 1] = 1                    # an entry above the diagonal, seen unless causal
    bm[t - 1, 0] = 0                    # and one below it hidden
    o, lse = oracle.attention_fwd(q, k, v, 0.8, causal=causal, kv_len=kv, block_mask=bm,
                                  block=bs)
    O, L = brute_force(q, k, v, 0.8, causal, kv, bm, bs)
    np.testing.assert_allclose(o, O, atol=1e-12)
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], L[fin], atol=1e-12)
    assert np.all(o[~fin] == 0)


def test_block_diagonal_mask_splits_the_sequence():
    """Only diagonal blocks kept: each block of rows attends only to its own
    keys, so the output equals attention run separately on each block."""
    rng = np.random.default_rng(70)
    B, H, N, d, bs = 1, 2, 20, 4, 6
    q, k, v = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    t = -(-N // bs)
    o, lse = oracle.attention_fwd(q, k, v, 0.5, block_mask=np.eye(t), block=bs)
    for r in range(t):
        sl = slice(r * bs, min((r + 1) * bs, N))
        o_r, l_r = oracle.attention_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.5)
        np.testing.assert_allclose(o[:, :, sl], o_r, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], l_r, atol=1e-13)


def test_lower_triangular_block_mask_is_causal_already():
    rng = np.random.default_rng(71)
    B, H, N, d, bs = 2, 2, 17, 3, 4
    q, k, v = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    t = -(-N // bs)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.6, causal=True)
    o2, l2 = oracle.attention_fwd(q, k, v, 0.6, causal=True, block_mask=np.tril(np.ones((t, t))),
                                  block=bs)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and the upper triangle alone leaves only the diagonal blocks' causal part
    o3, l3 = oracle.attention_fwd(q, k, v, 0.6, causal=True, block_mask=np.triu(np.ones((t, t))),
                                  block=bs)
    o4, l4 = oracle.attention_fwd(q, k, v, 0.6, causal=True, block_mask=np.eye(t), block=bs)
    np.testing.assert_array_equal(o3, o4)
    np.testing.assert_array_equal(l3, l4)


@pytest.mark.parametrize("causal,kv", [(False, None), (True, [8, 5])])
def test_backward_central_finite_differences(causal, kv):
    rng = np.random.default_rng(72)
    B, H, N, d, bs = 2, 2, 8, 3, 3
    q, do = rnd(rng, B, H, N, d), rnd(rng, B, H, N, d)
    k, v = rnd(rng, B, 1, N, d), rnd(rng, B, 1, N, d)
    t = -(-N // bs)
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]], dtype=np.uint8)[:t, :t]
    scale = 0.7
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, do, scale, causal=causal, kv_len=kv,
                                         block_mask=bm, block=bs)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal=causal, kv_len=kv, threads=1,
                                    block_mask=bm, block=bs)
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


def test_rejects_a_mask_of_the_wrong_shape():
    rng = np.random.default_rng(73)
    q = rnd(rng, 1, 1, 9, 2)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, q, q, 1.0, block_mask=np.ones((2, 2)), block=4)
