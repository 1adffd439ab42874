"""FP8 (E4M3) forward on the GPU.

The quantiser (fa_fp8_quantize) must write the same bytes and scales as the
oracle's quantisers (integer work: bit-exact).  The FP8 forward (fa_fwd_fp8)
is compared with the oracle's step-by-step FP8 algorithm run on the oracle's
own quantisation of the same bf16 inputs, with the O and LSE tolerances of
parity.py (the two differ only where fp32 and fp64 round a product or an
exponent differently, which can move a P onto the neighbouring E4M3 value).
A last check bounds the FP8 result against exact attention, the method's own
error, loosely."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref as F
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


def oracle_quantize(inp):
    q, k, v = (P.f64(inp[n]).astype(np.float32) for n in ("q", "k", "v"))
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    q8, sq = F.quantize_rows(q.reshape(B * H, N, d))
    k8, sk = F.quantize_rows(k.reshape(B * Hkv, N, d))
    v8t, sv = F.quantize_v_transposed(v.reshape(B * Hkv, N, d))
    return {"q8": q8.reshape(B, H, N, d), "q_scale": sq.reshape(B, H, -1),
            "k8": k8.reshape(B, Hkv, N, d), "k_scale": sk.reshape(B, Hkv, -1),
            "v8t": v8t.reshape(B, Hkv, d, -1), "v_scale": sv.reshape(B, Hkv)}


def run(w, inp):
    g = P.to_gpu(inp)
    o, lse, buf = fa.forward_fp8(g["q"], g["k"], g["v"], scale=w.scale, causal=w.causal,
                                 kv_len=g["kv_len"], window=w.window)
    fa.fa_check()
    return o, lse, buf


@pytest.mark.parametrize("B,H,Hkv,N,d", [(2, 4, 2, 300, 128), (1, 2, 2, 129, 256),
                                         (1, 3, 1, 1000, 128)])
def test_quantizer_is_bit_exact(B, H, Hkv, N, d):
    w = random_case(B, H, N, d, seed=N + d, h_kv=Hkv, qk_gain=2.0)
    inp = make_inputs(w, with_grad_out=False)
    g = P.to_gpu(inp)
    buf = fa.fp8_buffers(B, H, Hkv, N, d, "cuda")
    fa.fa_fp8_quantize(g["q"], g["k"], g["v"], buf)
    fa.fa_check()
    ref = oracle_quantize(inp)
    for name in ("q8", "k8", "v8t"):
        assert np.array_equal(buf[name].cpu().numpy(), ref[name]), name
    for name in ("q_scale", "k_scale", "v_scale"):
        assert np.array_equal(buf[name].cpu().numpy(), ref[name]), name


CASES = [
    # B, H, H_kv, N, d, causal, kv_len range, window
    (2, 2, 2, 300, 128, False, None, None),
    (1, 4, 2, 520, 128, True, None, None),
    (2, 2, 1, 257, 256, True, (100, 257), None),
    (1, 2, 2, 384, 256, False, None, None),
    (2, 3, 3, 129, 128, True, (1, 129), None),
    (1, 4, 1, 700, 128, True, None, (255, 0)),            # causal sliding window, MQA
    (2, 2, 2, 600, 128, False, (300, 600), (100, 200)),   # two-sided window, ragged lengths
    (1, 2, 1, 400, 256, True, None, (0, 0)),              # each query sees only its own key
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,kv,window", CASES)
def test_fp8_forward_against_oracle(B, H, Hkv, N, d, causal, kv, window):
    w = random_case(B, H, N, d, seed=3 * N + d, causal=causal, kv_len_range=kv, h_kv=Hkv,
                    window=window)
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    r = oracle_quantize(inp)
    kvn = None if inp["kv_len"] is None else inp["kv_len"].numpy()
    o_ref, lse_ref = F.attention_fp8(r["q8"], r["q_scale"], r["k8"], r["k_scale"], r["v8t"],
                                     r["v_scale"], w.scale, causal=causal, kv_len=kvn,
                                     window=window)
    P.check_o(P.f64(o), o_ref, w.name + " O (fp8)")
    P.check_lse(P.f64(lse), lse_ref, w.name + " LSE (fp8)")


def test_fp8_forward_near_exact_attention():
    """FP8's own error against exact attention of the bf16 inputs: a loose
    bound (E4M3 keeps 3 mantissa bits), checked on average and at worst."""
    w = random_case(1, 4, 1024, 128, seed=21, causal=True)
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    o_ref, lse_ref = oracle.attention_fwd(P.f64(inp["q"]), P.f64(inp["k"]), P.f64(inp["v"]),
                                          w.scale, causal=True)
    err = np.abs(P.f64(o) - o_ref)
    assert err.mean() <= 0.02 * np.abs(o_ref).max()
    assert err.max() <= 0.15 * np.abs(o_ref).max()
    assert np.abs(P.f64(lse) - lse_ref).max() <= 0.1


def test_fp8_long_sequence_sampled_rows():
    w = WORKLOADS["long_seq_b4_h32_n8192_d128_causal"]
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    b, h = 3, 31
    one = {k: (None if t is None else t[b:b + 1, h:h + 1].contiguous()) for k, t in inp.items()
           if k in ("q", "k", "v")}
    r = oracle_quantize(one)
    rows = [0, 1, 127, 128, 4095, 4096, 6000, 8191]
    o_ref, lse_ref = F.attention_fp8(r["q8"], r["q_scale"], r["k8"], r["k_scale"], r["v8t"],
                                     r["v_scale"], w.scale, causal=True, rows=rows)
    P.check_o(P.f64(o)[b:b + 1, h:h + 1, rows], o_ref[:, :, rows], w.name + " O (fp8)")
    P.check_lse(P.f64(lse)[b:b + 1, h:h + 1, rows], lse_ref[:, :, rows], w.name + " LSE (fp8)")
