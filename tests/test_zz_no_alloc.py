"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (an allocator hook that must not re-enter itself, a plugin that
only receives its tensors, a loop that cannot afford cudaMalloc's implicit
synchronisation) get the same gradients as fa_bwd without passing a
workspace; the library's own fixed scratch array stands in for it.  This file
sorts last so that a run stopping at the first failure has already run every
other test, and it passes both alone and after them.
"""
import pytest
import torch

from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import make_inputs, random_case

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fabuild.build()
    fa.load()


@pytest.mark.parametrize("B,H,N,d,causal,kv", [
    (2, 4, 384, 64, True, None),
    (3, 2, 300, 128, False, (100, 300)),
])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(B, H, N, d, causal, kv):
    w = random_case(B, H, N, d, seed=17 + N, causal=causal, kv_len_range=kv)
    g = P.to_gpu(make_inputs(w))
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=causal, kv_len=g["kv_len"])
    ref = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale, causal=causal,
                      kv_len=g["kv_len"])
    fa.fa_check()
    for call in range(2):
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        fa.fa_bwd_noalloc(g["q"], g["k"], g["v"], o, g["do"], lse, dq, dk, dv, w.scale,
                          causal, g["kv_len"])
        fa.fa_check()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            P.check_grad(P.f64(got), P.f64(want), f"call {call} {name}")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = fa.load()
    assert fa.fa_bwd_workspace_bytes(1, 1, 131072, 128) > 64 * 2 ** 20
    p = 0x1000
    st = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, 131072, 128, 0.088, 0, None, None)
    assert st == fa.FA_ERR_INVALID_ARG


def test_noalloc_large_call_then_small_ragged_call():
    """A small ragged problem right after a large one: the small call must not
    read what the large call left in the shared scratch (row statistics and
    the fp32 dQ accumulator past its own rows), so both must match fa_bwd."""
    shapes = [
        dict(B=2, H=8, N=4096, d=128, causal=True, kv=None, seed=41),   # 32.5 MiB of scratch
        dict(B=3, H=2, N=200, d=64, causal=False, kv=(50, 200), seed=42),
    ]
    for s in shapes:
        w = random_case(s["B"], s["H"], s["N"], s["d"], seed=s["seed"], causal=s["causal"],
                        kv_len_range=s["kv"])
        g = P.to_gpu(make_inputs(w))
        o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=w.causal,
                            kv_len=g["kv_len"])
        ref = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                          causal=w.causal, kv_len=g["kv_len"])
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        fa.fa_bwd_noalloc(g["q"], g["k"], g["v"], o, g["do"], lse, dq, dk, dv, w.scale,
                          w.causal, g["kv_len"])
        fa.fa_check()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            P.check_grad(P.f64(got), P.f64(want), f"N={s['N']} d={s['d']} {name}")
