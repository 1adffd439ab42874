"""Seeded synthetic inputs shaped like the pages' attention workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
draws random numbers and nothing else: it holds none of the attention
arithmetic, so the CPU oracle and the CUDA library can both be fed from it
without sharing any of the method.

Recipe (every tensor is drawn in fp32 on the CPU with ``torch.Generator``
seeded as stated, then rounded to bf16; the same bf16 bytes go to the GPU
and, widened exactly to float64, to the oracle):

* Q, K, V ~ iid N(0, 1), drawn in that order from one generator seeded with
  ``seed`` (Q with H heads, K and V with ``h_kv``); where ``qk_gain`` != 1 the
  fp32 Q and K are multiplied by it before rounding (the large-head-dimension
  workload uses 3, which makes the score standard deviation about 9 and
  stresses the max subtraction).
* dO ~ iid N(0, 1) from a generator seeded with ``seed + 100``.
* key-padding lengths ~ uniform integers in [lo, hi] (inclusive) from a
  generator seeded with ``seed + 200``.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    backward: bool
    qk_gain: float = 1.0
    kv_len_range: tuple = None     # (lo, hi) inclusive, or None for no padding
    h_kv: int = None               # K/V heads (grouped-query attention); None = H
    window: tuple = None           # flash-attn (left, right), -1 = unbounded; None = no window
    nq: int = None                 # decode: queries per head at the end of an N-key cache

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_heads(self) -> int:
        return self.H if self.h_kv is None else self.h_kv

    @property
    def queries(self) -> int:
        return self.N if self.nq is None else self.nq

    def visible_pairs(self) -> float:
        """(query, key) pairs one head computes: N^2, N^2/2 under the causal
        mask, and with a window the exact count of keys in each row's window
        (padding not discounted).  Decode: query t sits at position
        N - nq + t of the N-key cache."""
        N = self.N
        if self.nq is not None:
            wl, wr = self.window if self.window is not None else (-1, -1)
            total = 0
            for t in range(self.nq):
                pos = N - self.nq + t
                lo = 0 if wl < 0 else max(0, pos - wl)
                hi = N - 1 if wr < 0 else min(N - 1, pos + wr)
                if self.causal:
                    hi = min(hi, pos)
                total += max(0, hi - lo + 1)
            return float(total)
        if self.window is None:
            return N * N / 2 if self.causal else float(N * N)
        wl, wr = self.window
        total = 0
        for i in range(N):
            lo = 0 if wl < 0 else max(0, i - wl)
            hi = N - 1 if wr < 0 else min(N - 1, i + wr)
            if self.causal:
                hi = min(hi, i)
            total += max(0, hi - lo + 1)
        return float(total)

    def fwd_flops(self) -> float:
        """4*B*H*d per visible (query, key) pair: 4*B*H*N^2*d, halved under the
        causal mask (padding not discounted)."""
        return 4.0 * self.B * self.H * self.d * self.visible_pairs()

    def bwd_flops(self) -> float:
        """2.5 x the forward count."""
        return 2.5 * self.fwd_flops()


def _long_seq(N, causal):
    return Workload(f"long_seq_b{32768 // N}_h32_n{N}_d128_{'causal' if causal else 'full'}",
                    B=32768 // N, H=32, N=N, d=128, causal=causal, seed=3, backward=False)


WORKLOADS = {w.name: w for w in [
    Workload("single_head_b1_h1_n256_d64", 1, 1, 256, 64, causal=False, seed=0, backward=False),
    Workload("bert_large_b16_h16_n512_d64_pad", 16, 16, 512, 64, causal=False, seed=1,
             backward=True, kv_len_range=(256, 512)),
    Workload("gpt2_small_b8_h12_n1024_d64_causal", 8, 12, 1024, 64, causal=True, seed=2,
             backward=True),
    *[_long_seq(N, c) for N in (4096, 8192, 16384, 32768) for c in (False, True)],
    # head dimension 64 at a long sequence, forward and backward
    Workload("long_d64_b4_h16_n4096_full", 4, 16, 4096, 64, causal=False, seed=8,
             backward=True),
    Workload("large_head_b2_h16_n8192_d128_causal", 2, 16, 8192, 128, causal=True, seed=4,
             backward=True, qk_gain=3.0),
    Workload("large_head_b2_h16_n8192_d256_causal", 2, 16, 8192, 256, causal=True, seed=4,
             backward=True, qk_gain=3.0),
    # grouped-query attention, four query heads per K/V head (the GQA note of
    # the flash-attn API section names LLaMA 3 and Qwen)
    Workload("gqa_b2_h32_kv8_n8192_d128_causal", 2, 32, 8192, 128, causal=True, seed=5,
             backward=True, h_kv=8),
    # causal sliding window of 4096 keys (Mistral, per the sliding-window note)
    Workload("swa_b2_h32_n16384_d128_w4096_causal", 2, 32, 16384, 128, causal=True, seed=6,
             backward=True, window=(4095, 0)),
    # decoding one token per sequence against a 32K-key cache with four query
    # heads per K/V head (split-KV, the FlashDecoding note)
    Workload("decode_b4_h32_kv8_nq1_nk32768_d128", 4, 32, 32768, 128, causal=True, seed=7,
             backward=False, h_kv=8, nq=1),
]}


def make_inputs(w: Workload, with_grad_out: bool = None):
    """CPU tensors for workload ``w``: dict with q, k, v (bf16 [B,H,N,d]),
    optionally do (bf16) and kv_len (int32 [B] or None)."""
    shape = (w.B, w.H, w.queries, w.d)
    kv_shape = (w.B, w.kv_heads, w.N, w.d)
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    if w.qk_gain != 1.0:
        q.mul_(w.qk_gain)
        k.mul_(w.qk_gain)
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    del q, k, v
    if with_grad_out is None:
        with_grad_out = w.backward
    if with_grad_out:
        g2 = torch.Generator().manual_seed(w.seed + 100)
        out["do"] = torch.randn(shape, generator=g2, dtype=torch.float32).to(torch.bfloat16)
    out["kv_len"] = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        g3 = torch.Generator().manual_seed(w.seed + 200)
        out["kv_len"] = torch.randint(lo, hi + 1, (w.B,), generator=g3, dtype=torch.int32)
    return out


def random_case(B, H, N, d, seed, causal=False, kv_len_range=None, qk_gain=1.0, backward=True,
                h_kv=None, window=None):
    """An ad-hoc workload (edge-case tests) drawn with the same recipe."""
    return Workload(f"case_b{B}_h{H}_n{N}_d{d}", B, H, N, d, causal=causal, seed=seed,
                    backward=backward, qk_gain=qk_gain, kv_len_range=kv_len_range, h_kv=h_kv,
                    window=window)


def decode_case(B, H, h_kv, Nq, Nk, d, seed, causal=True, kv_len_range=None, window=None):
    """An ad-hoc decode workload: Nq queries per head, Nk keys."""
    return Workload(f"decode_b{B}_h{H}_kv{h_kv}_nq{Nq}_nk{Nk}_d{d}", B, H, Nk, d, causal=causal,
                    seed=seed, backward=False, kv_len_range=kv_len_range, h_kv=h_kv,
                    window=window, nq=Nq)


def make_decode_inputs(w: Workload):
    """q [B,H,Nq,d], k and v [B,H_kv,Nk,d], kv_len: make_inputs for a decode workload."""
    return make_inputs(w, with_grad_out=False)


def block_sparse_mask(T: int, seed: int = 0, band: int = 4, n_global: int = 2, n_random: int = 5):
    """A seeded [T, T] block mask (1 = computed) in the local + global + random
    pattern of long-context block-sparse attention: each 128-row query block
    sees the key blocks within `band` of its own, the first `n_global` key
    blocks and `n_random` others drawn at random; the first `n_global` query
    blocks see every key block.  About 25 % of the blocks at T = 64."""
    import numpy as np
    rng = np.random.default_rng(seed)
    bm = np.zeros((T, T), dtype=np.uint8)
    for a in range(T):
        bm[a, max(0, a - band): a + band + 1] = 1
        bm[a, :n_global] = 1
        bm[a, rng.choice(T, size=min(n_random, T), replace=False)] = 1
    bm[:n_global, :] = 1
    return bm
