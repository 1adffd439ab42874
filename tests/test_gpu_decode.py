"""Split-KV decoding on the GPU (fa_decode) against the fp64 oracle's
decode-shaped attention, with the O and LSE tolerances of parity.py."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import WORKLOADS, make_decode_inputs, decode_case

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fabuild.build()
    fa.load()


def run(w, inp, splits=None):
    g = P.to_gpu(inp)
    o, lse = fa.decode(g["q"], g["k"], g["v"], scale=w.scale, causal=w.causal,
                       kv_len=g["kv_len"], window=w.window, splits=splits)
    fa.fa_check()
    return o, lse


def compare(w, inp, o, lse, batches=None, kv_group=None):
    q, k, v = (P.f64(inp[n]) for n in ("q", "k", "v"))
    kv = None if inp["kv_len"] is None else inp["kv_len"].numpy()
    G = w.H // w.kv_heads
    bsel = slice(None) if batches is None else list(batches)
    if kv_group is None:
        hq, hk = slice(None), slice(None)
    else:
        hq, hk = slice(kv_group * G, (kv_group + 1) * G), slice(kv_group, kv_group + 1)
    o_ref, lse_ref = oracle.attention_decode(q[bsel][:, hq], k[bsel][:, hk], v[bsel][:, hk],
                                             w.scale, causal=w.causal,
                                             kv_len=None if kv is None else kv[bsel],
                                             window=w.window)
    P.check_o(P.f64(o)[bsel][:, hq], o_ref, w.name + " O")
    P.check_lse(P.f64(lse)[bsel][:, hq], lse_ref, w.name + " LSE")


CASES = [
    # B, H, H_kv, Nq, Nk, d, causal, kv_len range, window, splits
    (2, 8, 2, 1, 4099, 128, True, None, None, None),
    (1, 4, 4, 3, 1000, 64, True, (600, 1000), None, 3),
    (3, 32, 8, 4, 2500, 128, False, None, None, 5),
    (1, 2, 1, 1, 300, 256, True, None, None, 2),
    (2, 16, 1, 8, 777, 64, True, (5, 777), (100, -1), 2),
    (1, 8, 8, 16, 129, 128, False, None, None, 1),
    (2, 4, 2, 2, 5000, 256, True, (3000, 5000), (1000, 0), 4),
]


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,kv,win,splits", CASES)
def test_decode_against_oracle(B, H, Hkv, Nq, Nk, d, causal, kv, win, splits):
    w = decode_case(B, H, Hkv, Nq, Nk, d, seed=Nk + d, causal=causal, kv_len_range=kv, window=win)
    inp = make_decode_inputs(w)
    o, lse = run(w, inp, splits)
    compare(w, inp, o, lse)


def test_one_chunk_and_many_chunks_agree():
    w = decode_case(2, 8, 2, 2, 6000, 128, seed=7, causal=True)
    inp = make_decode_inputs(w)
    o1, lse1 = run(w, inp, 1)
    o2, lse2 = run(w, inp, 23)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (lse1 - lse2).abs().max().item() <= 1e-4
    compare(w, inp, o2, lse2)


def test_too_many_rows_per_kv_head_is_unsupported():
    q = torch.zeros(1, 32, 8, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.decode(q, k, k, splits=1)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


def test_decode_workload_sampled_group():
    w = WORKLOADS["decode_b4_h32_kv8_nq1_nk32768_d128"]
    inp = make_decode_inputs(w)
    o, lse = run(w, inp)
    compare(w, inp, o, lse, batches=[0, 3], kv_group=3)
