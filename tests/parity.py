"""Shared helpers for the GPU parity tests: run the library, run the oracle on
the same bf16 inputs (widened exactly to float64), compare with the stated
tolerances.

Tolerances (GPU bf16/fp32 outputs vs the fp64 oracle):
* O:   |dO_ij| <= 1e-2 + 2^-8 |O_ref,ij| for every element (the 2^-8 term is
       the largest relative error of rounding a value to bf16), and
       max|dO| <= 2e-2 max|O_ref|.
* LSE: max|dLSE| <= 1e-3.
* dQ, dK, dV: max|d| <= 2e-2 max|ref| + 1e-5 per tensor (the 1e-5 floor only
  matters when the exact gradient is identically zero, e.g. a single visible
  key, where fp32 rounding of dP - D leaves ~1e-7).
"""
import numpy as np
import torch

import oracle
from exact_attention_04_gb300 import fa

O_ABS = 1e-2
O_REL_ROUND = 2.0 ** -8
O_REL_MAX = 2e-2
LSE_ABS = 1e-3
GRAD_REL_MAX = 2e-2
GRAD_ABS_FLOOR = 1e-5


def f64(t):
    return t.detach().to("cpu", torch.float32).double().numpy()


def to_gpu(inputs):
    out = {}
    for k, t in inputs.items():
        out[k] = None if t is None else t.cuda()
    return out


def check_o(o_gpu, o_ref, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    bound = O_ABS + O_REL_ROUND * np.abs(o_ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: |dO|={err[worst]:.3e} > {bound[worst]:.3e} at {worst}"
    assert err.max() <= O_REL_MAX * np.abs(o_ref).max(), f"{what}: max|dO|={err.max():.3e}"
    return float(err.max())


def check_lse(lse_gpu, lse_ref, what=""):
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
    err = np.abs(lse_gpu[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err <= LSE_ABS, f"{what}: max|dLSE|={err:.3e}"
    return float(err)


def check_grad(g_gpu, g_ref, what=""):
    g_gpu = np.asarray(g_gpu, dtype=np.float64)
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite gradient"
    err = np.abs(g_gpu - g_ref).max()
    scale = np.abs(g_ref).max()
    assert err <= GRAD_REL_MAX * scale + GRAD_ABS_FLOOR, \
        f"{what}: max|d|={err:.3e} > {GRAD_REL_MAX} * {scale:.3e} + {GRAD_ABS_FLOOR}"
    return float(err / max(scale, 1e-30))


def gpu_forward(w, inp):
    g = to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=w.causal, kv_len=g["kv_len"])
    fa.fa_check()
    return g, o, lse


def gpu_backward(w, g, o, lse):
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                             causal=w.causal, kv_len=g["kv_len"])
    fa.fa_check()
    return dq, dk, dv


def heads(inp, b, h):
    """float64 [1,1,N,d] slices of one head."""
    return {k: (None if k == "kv_len" or t is None else f64(t[b:b + 1, h:h + 1]))
            for k, t in inp.items()}


def kv_of(inp, b):
    return None if inp["kv_len"] is None else [int(inp["kv_len"][b])]


def compare_forward_full(w, inp, o, lse, bh_list=None):
    """Whole-tensor (or per listed head) forward comparison."""
    if bh_list is None:
        o_ref, lse_ref = oracle.attention_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), w.scale,
                                              causal=w.causal, kv_len=inp["kv_len"])
        return check_o(f64(o), o_ref, w.name), check_lse(f64(lse), lse_ref, w.name)
    eo = el = 0.0
    for b, h in bh_list:
        x = heads(inp, b, h)
        o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], w.scale, causal=w.causal,
                                              kv_len=kv_of(inp, b))
        eo = max(eo, check_o(f64(o[b:b + 1, h:h + 1]), o_ref, f"{w.name} head {b},{h}"))
        el = max(el, check_lse(f64(lse[b:b + 1, h:h + 1]), lse_ref, f"{w.name} head {b},{h}"))
    return eo, el


def compare_forward_rows(w, inp, o, lse, bh_list, rows):
    """Forward comparison on chosen rows of chosen heads (large workloads)."""
    eo = el = 0.0
    for b, h in bh_list:
        q, k, v = (f64(inp[n][b, h]) for n in ("q", "k", "v"))
        kv = None if inp["kv_len"] is None else int(inp["kv_len"][b])
        o_ref, lse_ref = oracle.attention_fwd_rows(q, k, v, rows, w.scale, causal=w.causal, kv_len=kv)
        eo = max(eo, check_o(f64(o[b, h, rows]), o_ref, f"{w.name} head {b},{h}"))
        el = max(el, check_lse(f64(lse[b, h, rows]), lse_ref, f"{w.name} head {b},{h}"))
    return eo, el


def compare_backward(w, inp, grads, bh_list=None):
    dq, dk, dv = grads
    if bh_list is None:
        ref = oracle.attention_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]),
                                   w.scale, causal=w.causal, kv_len=inp["kv_len"])
        return [check_grad(f64(g), r, f"{w.name} {n}") for g, r, n in
                zip((dq, dk, dv), ref[:3], ("dQ", "dK", "dV"))]
    errs = [0.0, 0.0, 0.0]
    for b, h in bh_list:
        x = heads(inp, b, h)
        ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], w.scale, causal=w.causal,
                                   kv_len=kv_of(inp, b))
        for t, (g, r, n) in enumerate(zip((dq, dk, dv), ref[:3], ("dQ", "dK", "dV"))):
            errs[t] = max(errs[t], check_grad(f64(g[b:b + 1, h:h + 1]), r, f"{w.name} {n} head {b},{h}"))
    return errs


def sample_heads(B, H, k, seed=0):
    """(0,0), (B-1,H-1) and k-2 more distinct seeded heads."""
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (B - 1, H - 1)}
    while len(picks) < min(k, B * H):
        picks.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(picks)


def sample_rows(N, k=48, seed=0):
    """First/last rows, both sides of every few tile boundaries, and random rows."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, N - 1, N - 2, min(127, N - 1), min(128, N - 1), N // 2}
    rows |= set(int(r) for r in rng.integers(0, N, size=k))
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)
