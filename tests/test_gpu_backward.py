"""Backward parity on the GPU: dQ, dK, dV of libfa.so against the fp64 oracle."""
import numpy as np
import pytest
import torch

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


SMALL = [
    (1, 1, 128, 64, False, None),
    (2, 2, 383, 64, False, None),
    (2, 2, 383, 64, True, None),
    (1, 2, 129, 128, False, None),
    (2, 1, 300, 128, True, None),
    (3, 1, 333, 64, False, (1, 333)),
    (3, 2, 257, 128, True, (100, 257)),
    (1, 1, 1, 64, True, None),
    (1, 2, 17, 128, False, None),
    (2, 2, 320, 128, True, (200, 320)),
    (1, 2, 200, 256, True, None),
    (2, 1, 260, 256, False, (130, 260)),
    (1, 1, 64, 256, False, None),
    (2, 1, 129, 256, True, None),
]


@pytest.mark.parametrize("B,H,N,d,causal,kv", SMALL)
def test_backward_small_full_oracle(B, H, N, d, causal, kv):
    w = random_case(B, H, N, d, seed=N * 3 + d, causal=causal, kv_len_range=kv)
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    grads = P.gpu_backward(w, g, o, lse)
    P.compare_backward(w, inp, grads)


def test_backward_padded_keys_have_zero_gradient():
    w = random_case(2, 2, 300, 64, seed=5, causal=False, kv_len_range=(90, 200))
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    dq, dk, dv = P.gpu_backward(w, g, o, lse)
    for b in range(w.B):
        n = int(inp["kv_len"][b])
        assert torch.count_nonzero(dk[b, :, n:]) == 0
        assert torch.count_nonzero(dv[b, :, n:]) == 0


def test_backward_key_gradients_sum_to_zero():
    """Rows of dS sum to zero, so sum_j dK_j = 0 per head (up to bf16 rounding)."""
    w = random_case(1, 2, 512, 128, seed=9, causal=True)
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    dq, dk, dv = P.gpu_backward(w, g, o, lse)
    s = dk.float().sum(dim=2).abs().max().item()
    assert s <= 2e-2 * dk.float().abs().max().item() * 8


def test_bert_large_config_backward_sampled_heads():
    w = WORKLOADS["bert_large_b16_h16_n512_d64_pad"]
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    grads = P.gpu_backward(w, g, o, lse)
    errs = P.compare_backward(w, inp, grads, P.sample_heads(w.B, w.H, 6))
    print(f"{w.name}: rel errs dQ dK dV = {errs}")


def test_gpt2_config_backward_sampled_heads():
    w = WORKLOADS["gpt2_small_b8_h12_n1024_d64_causal"]
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    grads = P.gpu_backward(w, g, o, lse)
    errs = P.compare_backward(w, inp, grads, P.sample_heads(w.B, w.H, 4))
    print(f"{w.name}: rel errs dQ dK dV = {errs}")


def test_large_head_d128_config_backward_four_heads():
    """dQ, dK, dV of four seeded heads, always (0,0) and (B-1,H-1); the last
    head's key blocks run in the host-planned tail of the causal schedule."""
    w = WORKLOADS["large_head_b2_h16_n8192_d128_causal"]
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    grads = P.gpu_backward(w, g, o, lse)
    errs = P.compare_backward(w, inp, grads, P.sample_heads(w.B, w.H, 4, seed=128))
    print(f"{w.name}: rel errs dQ dK dV = {errs}")


def test_large_head_d256_config_backward_four_heads():
    """dQ, dK, dV of four seeded heads, always (0,0) and (B-1,H-1); the last
    head's key blocks run in the host-planned tail of the causal schedule."""
    w = WORKLOADS["large_head_b2_h16_n8192_d256_causal"]
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    grads = P.gpu_backward(w, g, o, lse)
    errs = P.compare_backward(w, inp, grads, P.sample_heads(w.B, w.H, 4, seed=256))
    print(f"{w.name}: rel errs dQ dK dV = {errs}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_padding_lengths_one_to_n_every_head(d):
    """Key lengths from 1 to N across six batch entries (tiles of 0 to 8 key
    blocks, 192 items on 152 SMs): every head against the oracle, forward
    and backward."""
    w = random_case(6, 4, 1000, d, seed=3 * d, causal=False, kv_len_range=(1, 1000))
    inp = make_inputs(w)
    inp["kv_len"][0], inp["kv_len"][1] = 1, 1000
    g, o, lse = P.gpu_forward(w, inp)
    P.compare_forward_full(w, inp, o, lse)
    P.compare_backward(w, inp, P.gpu_backward(w, g, o, lse))


@pytest.mark.parametrize("d,B,H,N,causal,kv,mask", [
    (64, 2, 4, 384, True, None, False), (64, 16, 16, 512, False, (256, 512), False),
    (64, 2, 8, 4096, False, None, True), (128, 2, 4, 2048, True, None, False),
    (256, 1, 4, 1024, True, None, False)])
def test_backward_is_deterministic(d, B, H, N, causal, kv, mask):
    """Reruns on the same inputs: dK and dV are each accumulated in tensor
    memory by one CTA, so they must agree bit for bit; dQ is summed across
    key blocks in L2 in an order that varies, so within a bf16 unit.  A race
    between the kernels' warps (the d = 64 kernel runs its warpgroups at
    different register counts) would show as bits that change between
    runs."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    w = random_case(B, H, N, d, seed=N + d, causal=causal, kv_len_range=kv)
    g = P.to_gpu(make_inputs(w))
    bm = torch.from_numpy(block_sparse_mask(-(-N // 128), seed=3)).cuda() if mask else None
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=causal, kv_len=g["kv_len"],
                        block_mask=bm)
    runs = [fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale, causal=causal,
                        kv_len=g["kv_len"], block_mask=bm) for _ in range(6)]
    fa.fa_check()
    dq0, dk0, dv0 = runs[0]
    for dq, dk, dv in runs[1:]:
        assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
        assert (dq.float() - dq0.float()).abs().max().item() <= 2 ** -7 * dq0.float().abs().max().item()


def test_long_d64_config_backward_four_heads():
    """Head dimension 64 at N = 4096: four seeded heads, always (0,0) and
    (B-1,H-1), every row."""
    w = WORKLOADS["long_d64_b4_h16_n4096_full"]
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    bh = P.sample_heads(w.B, w.H, 4, seed=w.N)
    P.compare_forward_full(w, inp, o, lse, bh)
    P.compare_backward(w, inp, P.gpu_backward(w, g, o, lse), bh)


def test_status_clean_after_runs():
    fa.fa_check()
