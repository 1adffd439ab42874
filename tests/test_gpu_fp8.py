"""FP8 (E4M3) forward on the GPU.

The quantiser (fa_fp8_quantize) must write the same bytes and scales as the
oracle's quantisers (integer work: bit-exact).  The FP8 forward (fa_fwd_fp8)
is compared, element by element, with EXACT attention (the fp64 oracle) of
the dequantised inputs q8*sq, k8*sk, v8*sv, under the bound of
parity.fp8_o_bound: it follows from E4M3's spacing alone (2^-4 relative for
a normal P operand, 2^-10 absolute below the normal range) and names none of
the kernel's choices (rescale slack, P multiplier), so any kernel that keeps
its P operands unsaturated and its reference rising must pass.  LSE adds
unrounded P, so it must match the exact LSE to 1e-3 as in the bf16 path.
"""
import numpy as np
import pytest
import torch

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


def check_fp8(w, inp, o, lse, bh_list=None, rows=None, block_mask=None):
    """Every listed head (all heads by default) of the E4M3 forward against
    exact attention of the oracle-quantised, dequantised inputs."""
    r = oracle_quantize(inp)
    B, H, N, _ = inp["q"].shape
    Hkv = inp["k"].shape[1]
    qd, kd, vd = P.dequantize(r, N)
    worst = 0.0
    for b, h in (bh_list or [(b, h) for b in range(B) for h in range(H)]):
        hk = h // (H // Hkv)
        kv = None if inp["kv_len"] is None else [int(inp["kv_len"][b])]
        og, lg = P.f64(o[b, h]), P.f64(lse[b, h])
        if rows is not None:
            og, lg = og[rows], lg[rows]
        worst = max(worst, P.check_fp8_head(og, lg, qd[b, h], kd[b, hk], vd[b, hk], w.scale,
                                            causal=w.causal, kv_len=kv, window=w.window,
                                            block_mask=block_mask, rows=rows,
                                            what=f"{w.name} head {b},{h} (fp8)"))
    return worst


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,kv,window", CASES)
def test_fp8_forward_against_exact_attention(B, H, Hkv, N, d, causal, kv, window):
    w = random_case(B, H, N, d, seed=3 * N + d, causal=causal, kv_len_range=kv, h_kv=Hkv,
                    window=window)
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    check_fp8(w, inp, o, lse)


def test_fp8_forward_large_scores_against_exact_attention():
    """Q and K scaled by 3, as in the large-head-dimension workload: scores of
    standard deviation about 9 put most P operands below E4M3's normal range
    and make the running maximum jump often (many O rescales)."""
    w = random_case(1, 4, 1024, 128, seed=21, causal=True, qk_gain=3.0)
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    check_fp8(w, inp, o, lse)


def test_fp8_long_sequence_sampled_rows():
    w = WORKLOADS["long_seq_b4_h32_n8192_d128_causal"]
    inp = make_inputs(w, with_grad_out=False)
    o, lse, _ = run(w, inp)
    rows = P.sample_rows(w.N, 40, seed=8)
    for b, h in P.sample_heads(w.B, w.H, 4, seed=8):
        sub = {n: inp[n][b:b + 1, h:h + 1].contiguous() for n in ("q", "k", "v")}
        sub["kv_len"] = None
        check_fp8(w, sub, o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], rows=rows)
