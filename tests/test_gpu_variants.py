"""Grouped K/V heads and sliding windows on the GPU: O, LSE, dQ, dK, dV of
libfa.so (fa_fwd_v / fa_bwd_v) against the fp64 oracle, with the tolerances
of parity.py."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import WORKLOADS, make_inputs, random_case

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fabuild.build()
    fa.load()


def run(w, inp, backward=True):
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=w.causal,
                        kv_len=g["kv_len"], window=w.window)
    fa.fa_check()
    grads = None
    if backward:
        grads = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                            causal=w.causal, kv_len=g["kv_len"], window=w.window)
        fa.fa_check()
    return o, lse, grads


def kv_len_np(inp):
    return None if inp["kv_len"] is None else inp["kv_len"].numpy()


def compare(w, inp, o, lse, grads, batches=None, kv_group=None):
    """Oracle on all heads, or on batch entries `batches` and the query heads
    of K/V head `kv_group` (with that K/V head alone)."""
    q, k, v = (P.f64(inp[n]) for n in ("q", "k", "v"))
    kv = kv_len_np(inp)
    G = w.H // w.kv_heads
    bsel = slice(None) if batches is None else list(batches)
    if kv_group is None:
        hq, hk = slice(None), slice(None)
    else:
        hq, hk = slice(kv_group * G, (kv_group + 1) * G), slice(kv_group, kv_group + 1)
    qs, ks, vs = q[bsel][:, hq], k[bsel][:, hk], v[bsel][:, hk]
    kvs = None if kv is None else kv[bsel]
    o_ref, lse_ref = oracle.attention_fwd(qs, ks, vs, w.scale, causal=w.causal, kv_len=kvs,
                                          window=w.window)
    P.check_o(P.f64(o)[bsel][:, hq], o_ref, w.name + " O")
    P.check_lse(P.f64(lse)[bsel][:, hq], lse_ref, w.name + " LSE")
    if grads is None:
        return
    do = P.f64(inp["do"])[bsel][:, hq]
    dq_ref, dk_ref, dv_ref, _ = oracle.attention_bwd(qs, ks, vs, do, w.scale, causal=w.causal,
                                                     kv_len=kvs, window=w.window)
    dq, dk, dv = grads
    P.check_grad(P.f64(dq)[bsel][:, hq], dq_ref, w.name + " dQ")
    P.check_grad(P.f64(dk)[bsel][:, hk], dk_ref, w.name + " dK")
    P.check_grad(P.f64(dv)[bsel][:, hk], dv_ref, w.name + " dV")


SMALL = [
    # B, H, H_kv, N, d, causal, kv_len range, window
    (2, 4, 2, 200, 64, False, None, (30, 50)),
    (1, 4, 1, 333, 128, True, None, (100, -1)),
    (2, 2, 2, 257, 128, False, (100, 257), (0, 0)),
    (1, 8, 2, 300, 256, True, (150, 300), (64, -1)),
    (2, 4, 4, 129, 64, False, None, (-1, 10)),
    (1, 2, 1, 520, 128, True, None, None),
    (2, 4, 2, 384, 256, False, None, (200, 100)),
    (1, 3, 1, 150, 64, True, (20, 60), (5, -1)),
    (2, 6, 3, 640, 128, False, (300, 640), (127, 129)),
    (1, 2, 2, 700, 64, True, None, (128, 0)),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,kv,win", SMALL)
def test_variant_small_full_oracle(B, H, Hkv, N, d, causal, kv, win):
    w = random_case(B, H, N, d, seed=N + d + H, causal=causal, kv_len_range=kv, h_kv=Hkv,
                    window=win)
    inp = make_inputs(w)
    o, lse, grads = run(w, inp)
    compare(w, inp, o, lse, grads)


def test_rows_that_see_no_key():
    """kv_len 20 with a left window of 5: queries from 26 on see no key, so
    O = 0, LSE = -inf, and their dQ is 0; keys past kv_len get dK = dV = 0."""
    w = random_case(1, 2, 200, 64, seed=3, causal=True, kv_len_range=(20, 20), window=(5, -1))
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = run(w, inp)
    assert torch.all(torch.isneginf(lse[0, :, 26:]))
    assert torch.count_nonzero(o[0, :, 26:]) == 0
    assert torch.count_nonzero(dq[0, :, 26:]) == 0
    assert torch.count_nonzero(dk[0, :, 20:]) == 0 and torch.count_nonzero(dv[0, :, 20:]) == 0
    compare(w, inp, o, lse, (dq, dk, dv))


def test_gqa_equals_repeated_kv_on_gpu():
    """The GPU's GQA forward equals its MHA forward on K/V heads repeated
    across each group (the same kernels on the same keys: bit-exact)."""
    w = random_case(2, 8, 512, 128, seed=11, causal=True, h_kv=2)
    inp = make_inputs(w)
    o, lse, _ = run(w, inp, backward=False)
    g = P.to_gpu(inp)
    kr = g["k"].repeat_interleave(4, dim=1).contiguous()
    vr = g["v"].repeat_interleave(4, dim=1).contiguous()
    o2, lse2 = fa.forward(g["q"], kr, vr, scale=w.scale, causal=True)
    fa.fa_check()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_gqa_workload_sampled_group():
    w = WORKLOADS["gqa_b2_h32_kv8_n8192_d128_causal"]
    inp = make_inputs(w)
    o, lse, grads = run(w, inp)
    compare(w, inp, o, lse, grads, batches=[1], kv_group=7)


def test_sliding_window_workload_sampled_heads():
    w = WORKLOADS["swa_b2_h32_n16384_d128_w4096_causal"]
    inp = make_inputs(w)
    o, lse, grads = run(w, inp)
    compare(w, inp, o, lse, grads, batches=[0], kv_group=31)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_window_of_one_key_is_exact(d):
    """Window (0, 0): every query sees only its own key, so P = 1 exactly:
    O must equal V bit for bit, LSE = scale q_i.k_i, dV = dO bit for bit, and
    dQ, dK vanish up to fp32 rounding of dP - D.  (A row maximum taken over
    more than the row's own scores shows up here as O != V.)"""
    w = random_case(2, 2, 300, d, seed=d, causal=False, window=(0, 0))
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = run(w, inp)
    g = P.to_gpu(inp)
    assert torch.equal(o, g["v"])
    assert torch.equal(dv, g["do"])
    s_ii = w.scale * (P.f64(inp["q"]) * P.f64(inp["k"])).sum(-1)
    assert np.abs(P.f64(lse) - s_ii).max() <= 1e-5
    assert dq.float().abs().max().item() <= 1e-3
    assert dk.float().abs().max().item() <= 1e-3
