"""Shared helpers for the GPU parity tests: run the library, run the oracle on
the same bf16 inputs (widened exactly to float64), compare with the stated
tolerances.

Tolerances (GPU bf16/fp32 outputs vs the fp64 oracle):
* O:   |dO_ij| <= 1e-2 + 2^-8 |O_ref,ij| for every element (the 2^-8 term is
       the largest relative error of rounding a value to bf16), and
       max|dO| <= 2e-2 max|O_ref|.  The kernels round P to bf16 before the
       P V product ("4. FlashAttention 深度剖析" 4.7.3 casts p to V's type),
       which moves each weight by up to 2^-8 of itself while the row sum
       adds the unrounded p; so an element may also move by
       2^-8 sum_k P_ik |V_kj|.  Where the first bound fails, that term is
       computed from the oracle (attention of |V|) and added.
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


P_REL_ROUND = 2.0 ** -8


def check_o(o_gpu, o_ref, what="", abs_v_attention=None):
    """abs_v_attention: None, or a callable returning sum_k P_ik |V_kj| (exact
    attention of |V|, the oracle's) shaped like o_ref; it is called only when
    the bound without the P-rounding term fails somewhere."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    bound = O_ABS + O_REL_ROUND * np.abs(o_ref)
    if abs_v_attention is not None and not np.all(err <= bound):
        bound = bound + P_REL_ROUND * np.asarray(abs_v_attention(), dtype=np.float64)
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
        q, k, v = f64(inp["q"]), f64(inp["k"]), f64(inp["v"])
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, causal=w.causal,
                                              kv_len=inp["kv_len"])
        av = lambda: oracle.attention_fwd(q, k, np.abs(v), w.scale, causal=w.causal,  # noqa: E731
                                          kv_len=inp["kv_len"])[0]
        return check_o(f64(o), o_ref, w.name, av), check_lse(f64(lse), lse_ref, w.name)
    eo = el = 0.0
    for b, h in bh_list:
        x = heads(inp, b, h)
        o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], w.scale, causal=w.causal,
                                              kv_len=kv_of(inp, b))
        av = lambda x=x, b=b: oracle.attention_fwd(x["q"], x["k"], np.abs(x["v"]), w.scale,  # noqa: E731
                                                   causal=w.causal, kv_len=kv_of(inp, b))[0]
        eo = max(eo, check_o(f64(o[b:b + 1, h:h + 1]), o_ref, f"{w.name} head {b},{h}", av))
        el = max(el, check_lse(f64(lse[b:b + 1, h:h + 1]), lse_ref, f"{w.name} head {b},{h}"))
    return eo, el


def compare_forward_rows(w, inp, o, lse, bh_list, rows):
    """Forward comparison on chosen rows of chosen heads (large workloads)."""
    eo = el = 0.0
    for b, h in bh_list:
        q, k, v = (f64(inp[n][b, h]) for n in ("q", "k", "v"))
        kv = None if inp["kv_len"] is None else int(inp["kv_len"][b])
        o_ref, lse_ref = oracle.attention_fwd_rows(q, k, v, rows, w.scale, causal=w.causal, kv_len=kv)
        av = lambda q=q, k=k, v=v, kv=kv: oracle.attention_fwd_rows(  # noqa: E731
            q, k, np.abs(v), rows, w.scale, causal=w.causal, kv_len=kv)[0]
        eo = max(eo, check_o(f64(o[b, h, rows]), o_ref, f"{w.name} head {b},{h}", av))
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


# ---------------------------------------------------------------------------
# FP8 (E4M3) forward.  The reference is exact attention (the fp64 oracle) of
# the DEQUANTISED inputs qd = q8*sq, kd = k8*sk, vd = v8*sv, which are the
# values the E4M3 kernel multiplies.  What separates the kernel's O from it
# is the rounding of P to E4M3 before the P.V product ("4. FlashAttention
# 深度剖析" 4.5.4: E4M3 operands, fp32 accumulation), plus fp32 arithmetic.
#
# Bound.  Let w_j be the exact weights of a row and w_max their maximum.  A
# kernel feeds x_j = c_b * w_j * l (its operand for key j: some multiplier
# times the weight against its running normaliser l) to E4M3 and divides the
# P.V sum by the same c*l it summed from the UNROUNDED p.  E4M3 rounds a
# normal x (>= 2^-6) to within half a quantum, at most 2^-4 * x, and a
# subnormal x to within min(x, 2^-10).  Provided (i) the row's largest
# operand is at least 1 at the final reference (the kernel's reference never
# exceeds the row maximum, and its multiplier is >= 1), (ii) the reference
# never moves down, and (iii) no operand exceeds 448 (no saturation), the
# error of weight j after normalisation is at most
#     e_j = max(2^-4 w_j, min(w_j, 2^-10 w_max)),
# so |O_gpu - O_exact| <= sum_j e_j |vd_j| elementwise, plus fp32 rounding of
# the scores, the exponentials and the sums (FP8_FP32_REL of sum_j w_j |vd_j|)
# and bf16's rounding of the stored O (2^-8 relative).  Nothing in it names
# the kernel's slack or multiplier: any choice that satisfies (i)-(iii)
# passes.  LSE = m + ln l adds unrounded p, so it must match the exact LSE
# to LSE_ABS like the bf16 path.
# ---------------------------------------------------------------------------
FP8_P_REL = 2.0 ** -4          # half an E4M3 quantum, relative, normal values
FP8_P_SUB = 2.0 ** -10         # half the E4M3 subnormal spacing 2^-9, absolute
FP8_FP32_REL = 4e-3            # fp32 scores (|s| < ~200), exp2, sums over <= 32768 keys


def dequantize(r, N):
    """qd, kd, vd (float64 [B,H,N,d] / [B,H_kv,N,d]) from E4M3 codes and scales
    as the oracle's quantisers write them (q8, q_scale, k8, k_scale, v8t,
    v_scale)."""
    from oracle import fp8_ref as F
    qd = F.e4m3_decode(r["q8"]) * np.repeat(r["q_scale"], 128, axis=2)[:, :, :N, None]
    kd = F.e4m3_decode(r["k8"]) * np.repeat(r["k_scale"], 128, axis=2)[:, :, :N, None]
    vd = (F.e4m3_decode(r["v8t"][..., :N]).transpose(0, 1, 3, 2)
          * r["v_scale"][:, :, None, None])
    return qd, kd, vd


def oracle_weights(q, k, scale, causal=False, kv_len=None, window=None, block_mask=None,
                   rows=None):
    """Exact attention weights P [len(rows) or N, N] of one head (q, k float64
    [N, d]) as the oracle computes them: O = P V with V one-hot over a chunk
    of d keys gives P's columns of that chunk, masks included."""
    N, d = q.shape
    rows_arr = np.arange(N) if rows is None else np.asarray(rows)
    Pm = np.zeros((rows_arr.size, N))
    for c0 in range(0, N, d):
        n = min(d, N - c0)
        onehot = np.zeros((N, d))
        onehot[c0 + np.arange(n), np.arange(n)] = 1.0
        if rows is None:
            o, _ = oracle.attention_fwd(q[None, None], k[None, None], onehot[None, None], scale,
                                        causal=causal, kv_len=kv_len, window=window,
                                        block_mask=block_mask)
            o = o[0, 0]
        else:
            assert block_mask is None
            o, _ = oracle.attention_fwd_rows(q, k, onehot, rows_arr, scale, causal=causal,
                                             kv_len=None if kv_len is None else kv_len[0],
                                             window=window)
        Pm[:, c0:c0 + n] = o[:, :n]
    return Pm


def fp8_o_bound(Pw, vd, o_ref):
    """Elementwise bound on |O_fp8 - O_exact| for weights Pw [R, N], values vd
    [N, d] and the exact O [R, d] (see the derivation above)."""
    wmax = Pw.max(axis=1, keepdims=True)
    e = np.maximum(FP8_P_REL * Pw, np.minimum(Pw, FP8_P_SUB * wmax))
    av = np.abs(vd)
    body = e @ av + FP8_FP32_REL * (Pw @ av)
    return body * (1 + O_REL_ROUND) + O_REL_ROUND * np.abs(o_ref) + 1e-6


def check_fp8_head(o_gpu, lse_gpu, qd, kd, vd, scale, causal=False, kv_len=None, window=None,
                   block_mask=None, rows=None, what=""):
    """One head: O and LSE of the E4M3 forward (rows of it, if given) against
    exact attention of the dequantised inputs (qd, kd, vd [N, d])."""
    if rows is None:
        o_ref, lse_ref = oracle.attention_fwd(qd[None, None], kd[None, None], vd[None, None],
                                              scale, causal=causal, kv_len=kv_len,
                                              window=window, block_mask=block_mask)
        o_ref, lse_ref = o_ref[0, 0], lse_ref[0, 0]
    else:
        o_ref, lse_ref = oracle.attention_fwd_rows(qd, kd, vd, rows, scale, causal=causal,
                                                   kv_len=None if kv_len is None else kv_len[0],
                                                   window=window)
    Pw = oracle_weights(qd, kd, scale, causal=causal, kv_len=kv_len, window=window,
                        block_mask=block_mask, rows=rows)
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    bound = fp8_o_bound(Pw, vd, o_ref)
    err = np.abs(o_gpu - o_ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), \
        f"{what}: |dO|={err[worst]:.3e} > E4M3 bound {bound[worst]:.3e} at {worst}"
    check_lse(lse_gpu, lse_ref, what)
    return float((err / bound).max())
