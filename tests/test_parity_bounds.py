"""CPU checks of the forward parity bound in tests/parity.py (no GPU needed).

The kernels round P to bf16 before the P V product ("4. FlashAttention 深度
剖析" 4.7.3 casts p to V's type) while the row sum adds the unrounded p.
Rounding a weight to bf16 (8 significant bits) moves it by up to 2^-8 of
itself, so an output element can move by up to 2^-8 sum_k P_ik |V_kj| on
top of the final rounding of O to bf16.  This file builds the worst case on
purpose, with a plain emulation of those two roundings against the fp64
oracle: the bound without the P term fails, the full bound holds.
"""
import numpy as np
import torch

import oracle
import parity as P


def bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def emulate(q, k, v, scale, ref_below_max):
    """O with P = exp(s - m) rounded to bf16, m = row max - ref_below_max,
    the row sum of unrounded p, and O rounded to bf16."""
    s = (q @ k.T) * scale
    m = s.max(axis=1, keepdims=True) - ref_below_max
    p = np.exp(s - m)
    return bf16((bf16(p) @ v) / p.sum(axis=1, keepdims=True))


def test_p_rounding_term_is_needed_and_sufficient():
    # query row 0 sees one dominant key (score 5 against -5 for 127 others,
    # weight 0.994) whose value -4.5 sits where bf16's spacing is 2^-5, and
    # the reference lies 3.05 octaves below the row maximum, where rounding
    # the dominant p to bf16 pushes O onto the far side of a bf16 midpoint
    d = 8
    q = np.zeros((128, d)); q[0, 0] = 1.0
    k = np.full((128, d), 0.0); k[:, 0] = -5.0; k[0, 0] = 5.0
    v = np.full((128, d), 0.8); v[0, :] = -4.5
    o_ref, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0)
    av = oracle.attention_fwd(q[None, None], k[None, None], np.abs(v)[None, None], 1.0)[0]
    o = emulate(q, k, v, 1.0, np.log(2.0) * 3.05)
    err = np.abs(o[0] - o_ref[0, 0, 0])
    base = P.O_ABS + P.O_REL_ROUND * np.abs(o_ref[0, 0, 0])
    assert np.any(err > base), "the case should need the P-rounding term"
    assert np.all(err <= base + P.P_REL_ROUND * av[0, 0, 0])


def test_p_rounding_bound_holds_on_random_peaked_rows():
    rng = np.random.default_rng(7)
    for _ in range(4):
        N, d = 384, 64
        q = bf16(rng.standard_normal((N, d)) * 3)
        k = bf16(rng.standard_normal((N, d)) * 3)
        v = bf16(rng.standard_normal((N, d)) * 2)
        scale = 1 / np.sqrt(d)
        o_ref, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale)
        av = oracle.attention_fwd(q[None, None], k[None, None], np.abs(v)[None, None], scale)[0]
        for ref_below in (0.0, 6.0, 16.0):
            o = emulate(q, k, v, scale, ref_below)
            P.check_o(o[None, None], o_ref, "emulated bf16 P", lambda: av)
