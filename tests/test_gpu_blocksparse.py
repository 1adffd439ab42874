"""Block-sparse attention on the GPU: a [ceil(N/128)]^2 block mask whose zero
entries the kernels skip (Block-Sparse FlashAttention, "炉案与百步之外的仓库…"
第八部分), against the oracle with the same mask, element by element, with
the parity tolerances of parity.py."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref as F
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


def random_mask(T, density, seed, empty_row=None):
    rng = np.random.default_rng(seed)
    bm = (rng.random((T, T)) < density).astype(np.uint8)
    if empty_row is not None:
        bm[empty_row] = 0                     # a query block that sees no key at all
    return bm


CASES = [
    # B, H, H_kv, N, d, causal, kv_len range, density, empty row
    (2, 2, 2, 700, 128, False, None, 0.5, None),
    (1, 4, 2, 1000, 128, True, None, 0.6, 2),
    (2, 2, 1, 520, 64, False, (300, 520), 0.5, None),
    (1, 2, 2, 640, 256, True, None, 0.7, None),
    (2, 3, 3, 383, 64, True, (100, 383), 0.4, 1),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,kv,density,empty", CASES)
def test_forward_block_mask_against_oracle(B, H, Hkv, N, d, causal, kv, density, empty):
    w = random_case(B, H, N, d, seed=N + d, causal=causal, kv_len_range=kv, h_kv=Hkv,
                    backward=False)
    inp = make_inputs(w, with_grad_out=False)
    T = -(-N // 128)
    bm = random_mask(T, density, seed=N, empty_row=empty)
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=causal, kv_len=g["kv_len"],
                        block_mask=torch.from_numpy(bm).cuda())
    fa.fa_check()
    kvn = None if inp["kv_len"] is None else inp["kv_len"].numpy()
    o_ref, lse_ref = oracle.attention_fwd(P.f64(inp["q"]), P.f64(inp["k"]), P.f64(inp["v"]),
                                          w.scale, causal=causal, kv_len=kvn, block_mask=bm)
    P.check_o(P.f64(o), o_ref, w.name + " O (block mask)")
    P.check_lse(P.f64(lse), lse_ref, w.name + " LSE (block mask)")
    if empty is not None:
        rows = slice(empty * 128, min((empty + 1) * 128, N))
        assert torch.all(o[:, :, rows] == 0)
        assert torch.all(torch.isinf(lse[:, :, rows]) & (lse[:, :, rows] < 0))


def test_full_mask_equals_no_mask_bit_for_bit():
    w = random_case(2, 2, 900, 128, seed=5, causal=True, backward=False)
    g = P.to_gpu(make_inputs(w, with_grad_out=False))
    T = -(-900 // 128)
    o1, l1 = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=False, window=(-1, 0))
    o2, l2 = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=True,
                        block_mask=torch.ones(T, T, dtype=torch.uint8, device="cuda"))
    fa.fa_check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("N,d,causal", [(600, 128, False), (520, 256, True)])
def test_fp8_forward_block_mask_against_oracle(N, d, causal):
    w = random_case(1, 2, N, d, seed=3 * N, causal=causal, backward=False)
    inp = make_inputs(w, with_grad_out=False)
    T = -(-N // 128)
    bm = random_mask(T, 0.6, seed=N + 1)
    g = P.to_gpu(inp)
    o, lse, _ = fa.forward_fp8(g["q"], g["k"], g["v"], scale=w.scale, causal=causal,
                               block_mask=torch.from_numpy(bm).cuda())
    fa.fa_check()
    q, k, v = (P.f64(inp[n]).astype(np.float32) for n in ("q", "k", "v"))
    q8, sq = F.quantize_rows(q.reshape(2, N, d))
    k8, sk = F.quantize_rows(k.reshape(2, N, d))
    v8t, sv = F.quantize_v_transposed(v.reshape(2, N, d))
    r = {"q8": q8.reshape(1, 2, N, d), "q_scale": sq.reshape(1, 2, -1),
         "k8": k8.reshape(1, 2, N, d), "k_scale": sk.reshape(1, 2, -1),
         "v8t": v8t.reshape(1, 2, d, -1), "v_scale": sv.reshape(1, 2)}
    qd, kd, vd = P.dequantize(r, N)
    for h in range(2):
        P.check_fp8_head(P.f64(o[0, h]), P.f64(lse[0, h]), qd[0, h], kd[0, h], vd[0, h],
                         w.scale, causal=causal, block_mask=bm,
                         what=f"{w.name} head {h} (fp8, block mask)")




BWD_CASES = [
    # B, H, H_kv, N, d, causal, kv_len range, density, empty row
    (2, 2, 2, 520, 128, False, None, 0.5, None),
    (1, 4, 2, 700, 128, True, None, 0.6, 1),
    (2, 2, 1, 383, 64, True, (100, 383), 0.5, None),
    (1, 2, 2, 640, 64, False, None, 0.4, 2),
    (1, 2, 1, 520, 256, True, None, 0.7, None),
    (2, 1, 1, 300, 256, False, (150, 300), 0.5, 0),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,kv,density,empty", BWD_CASES)
def test_backward_block_mask_against_oracle(B, H, Hkv, N, d, causal, kv, density, empty):
    w = random_case(B, H, N, d, seed=2 * N + d, causal=causal, kv_len_range=kv, h_kv=Hkv)
    inp = make_inputs(w)
    T = -(-N // 128)
    bm = random_mask(T, density, seed=N + 7, empty_row=empty)
    bm_gpu = torch.from_numpy(bm).cuda()
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=causal, kv_len=g["kv_len"],
                        block_mask=bm_gpu)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                             causal=causal, kv_len=g["kv_len"], block_mask=bm_gpu)
    fa.fa_check()
    kvn = None if inp["kv_len"] is None else inp["kv_len"].numpy()
    dq_r, dk_r, dv_r, _ = oracle.attention_bwd(P.f64(inp["q"]), P.f64(inp["k"]), P.f64(inp["v"]),
                                               P.f64(inp["do"]), w.scale, causal=causal,
                                               kv_len=kvn, block_mask=bm)
    P.check_grad(P.f64(dq), dq_r, w.name + " dQ (block mask)")
    P.check_grad(P.f64(dk), dk_r, w.name + " dK (block mask)")
    P.check_grad(P.f64(dv), dv_r, w.name + " dV (block mask)")


def test_backward_key_block_with_no_query_has_zero_gradient():
    """A key block whose column of the mask is all zero meets no query: its dK
    and dV must be exactly zero (the kernels write them without a step)."""
    w = random_case(1, 2, 512, 128, seed=77, causal=False)
    inp = make_inputs(w)
    bm = np.ones((4, 4), dtype=np.uint8)
    bm[:, 2] = 0
    bm_gpu = torch.from_numpy(bm).cuda()
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, block_mask=bm_gpu)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                             block_mask=bm_gpu)
    fa.fa_check()
    assert torch.all(dk[:, :, 256:384] == 0) and torch.all(dv[:, :, 256:384] == 0)
    assert dk[:, :, :256].abs().max() > 0


def test_blocksparse_bench_workload_sampled_heads():
    """The bench's block-sparse workload (B=2, H=16, N=8192, d=128, the local +
    global + random pattern at about 25 % density), two heads against the
    oracle, forward and backward, in the launch configuration the bench times
    (the mask with its host copy, so the schedule is the balanced one)."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    w = random_case(2, 16, 8192, 128, seed=12, causal=False)
    inp = make_inputs(w)
    bm = block_sparse_mask(64, seed=12)
    bm_gpu = fa.BlockMask(bm)
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, block_mask=bm_gpu)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                             block_mask=bm_gpu)
    fa.fa_check()
    for b, h in ((0, 0), (1, 15)):
        one = {n: inp[n][b:b + 1, h:h + 1] for n in ("q", "k", "v", "do")}
        o_r, l_r = oracle.attention_fwd(P.f64(one["q"]), P.f64(one["k"]), P.f64(one["v"]),
                                        w.scale, block_mask=bm)
        P.check_o(P.f64(o[b:b + 1, h:h + 1]), o_r, f"block-sparse O ({b},{h})")
        P.check_lse(P.f64(lse[b:b + 1, h:h + 1]), l_r, f"block-sparse LSE ({b},{h})")
        dq_r, dk_r, dv_r, _ = oracle.attention_bwd(P.f64(one["q"]), P.f64(one["k"]),
                                                   P.f64(one["v"]), P.f64(one["do"]), w.scale,
                                                   block_mask=bm)
        P.check_grad(P.f64(dq[b:b + 1, h:h + 1]), dq_r, f"block-sparse dQ ({b},{h})")
        P.check_grad(P.f64(dk[b:b + 1, h:h + 1]), dk_r, f"block-sparse dK ({b},{h})")
        P.check_grad(P.f64(dv[b:b + 1, h:h + 1]), dv_r, f"block-sparse dV ({b},{h})")


@pytest.mark.parametrize("d,causal,window", [(128, False, (200, 50)), (64, True, (300, 0))])
def test_block_mask_with_window_forward_and_backward(d, causal, window):
    """The window bounds each tile's block range and the block mask then drops
    blocks inside it; both together against the oracle with both masks."""
    N = 900
    w = random_case(2, 2, N, d, seed=N + d, causal=causal, window=window)
    inp = make_inputs(w)
    T = -(-N // 128)
    bm = random_mask(T, 0.6, seed=d)
    bm_gpu = torch.from_numpy(bm).cuda()
    g = P.to_gpu(inp)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=causal, window=window,
                        block_mask=bm_gpu)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                             causal=causal, window=window, block_mask=bm_gpu)
    fa.fa_check()
    args = [P.f64(inp[n]) for n in ("q", "k", "v")]
    o_r, l_r = oracle.attention_fwd(*args, w.scale, causal=causal, window=window, block_mask=bm)
    P.check_o(P.f64(o), o_r, "O (window + block mask)")
    P.check_lse(P.f64(lse), l_r, "LSE (window + block mask)")
    dq_r, dk_r, dv_r, _ = oracle.attention_bwd(*args, P.f64(inp["do"]), w.scale, causal=causal,
                                               window=window, block_mask=bm)
    P.check_grad(P.f64(dq), dq_r, "dQ (window + block mask)")
    P.check_grad(P.f64(dk), dk_r, "dK (window + block mask)")
    P.check_grad(P.f64(dv), dv_r, "dV (window + block mask)")


@pytest.mark.parametrize("d,Hkv,window", [(128, 16, None), (256, 16, None), (64, 16, None),
                                          (128, 4, (-1, 0))])
def test_host_and_device_planned_schedules_agree(d, Hkv, window):
    """With the mask's host copy the launch plans a balanced tail of tiles and
    key blocks; without it each CTA sorts the tiles (and the backward's
    planning kernel the key blocks) by cost on the device and takes its
    items in the turning deal.  A tile's, or a key block's, arithmetic does
    not depend on the SM that runs it, so O, LSE, dK and dV agree bit for
    bit; dQ is summed across key blocks in L2 in an order that varies, so it
    agrees within a bf16 unit.  A tile or key block either plan missed or ran
    twice would show here (at N = 8192 the host plan has a tail of 14 heads
    on 152 SMs, the device deal 14 rounds)."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    w = random_case(2, 16, 8192, d, seed=d + Hkv, causal=False, h_kv=Hkv)
    g = P.to_gpu(make_inputs(w))
    bm = block_sparse_mask(64, seed=12)
    plain, balanced = torch.from_numpy(bm).cuda(), fa.BlockMask(bm)
    out = []
    for m in (plain, balanced):
        o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, window=window, block_mask=m)
        grads = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                            window=window, block_mask=m)
        out.append((o, lse) + tuple(grads))
    fa.fa_check()
    (o1, l1, dq1, dk1, dv1), (o2, l2, dq2, dk2, dv2) = out
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    diff = (dq1.float() - dq2.float()).abs().max().item()
    assert diff <= 2 ** -7 * dq1.float().abs().max().item(), diff
    assert (dq1 != dq2).float().mean().item() < 0.01


@pytest.mark.parametrize("d", [128, 256])
def test_host_and_device_planned_schedules_agree_fp8(d):
    """The E4M3 forward with and without the mask's host copy (the host-planned
    tail, the device's cost-sorted deal): the same tiles with the same
    arithmetic, so O and LSE agree bit for bit."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    w = random_case(2, 16, 8192, d, seed=d + 7, causal=False)
    g = P.to_gpu(make_inputs(w))
    bm = block_sparse_mask(64, seed=3)
    o1, l1, _ = fa.forward_fp8(g["q"], g["k"], g["v"], scale=w.scale,
                               block_mask=torch.from_numpy(bm).cuda())
    o2, l2, _ = fa.forward_fp8(g["q"], g["k"], g["v"], scale=w.scale, block_mask=fa.BlockMask(bm))
    fa.fa_check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_balanced_schedule_with_padding_against_oracle():
    """Key padding with the balanced schedule (the plan counts blocks over the
    full length; the kernels still stop at each entry's kv_len), two heads
    against the oracle."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    N = 4000
    w = random_case(2, 8, N, 128, seed=41, causal=False, kv_len_range=(1500, N))
    inp = make_inputs(w)
    T = -(-N // 128)
    bm = block_sparse_mask(T, seed=4, band=2, n_random=3)
    g = P.to_gpu(inp)
    kv = g.get("kv_len")
    m = fa.BlockMask(bm)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, kv_len=kv, block_mask=m)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale, kv_len=kv,
                             block_mask=m)
    fa.fa_check()
    kvl = None if inp.get("kv_len") is None else [int(x) for x in inp["kv_len"]]
    for b, h in ((0, 3), (1, 6)):
        one = {n: inp[n][b:b + 1, h:h + 1] for n in ("q", "k", "v", "do")}
        kl = None if kvl is None else [kvl[b]]
        o_r, l_r = oracle.attention_fwd(P.f64(one["q"]), P.f64(one["k"]), P.f64(one["v"]),
                                        w.scale, kv_len=kl, block_mask=bm)
        P.check_o(P.f64(o[b:b + 1, h:h + 1]), o_r, f"padded block-sparse O ({b},{h})")
        P.check_lse(P.f64(lse[b:b + 1, h:h + 1]), l_r, f"padded block-sparse LSE ({b},{h})")
        dq_r, dk_r, dv_r, _ = oracle.attention_bwd(P.f64(one["q"]), P.f64(one["k"]),
                                                   P.f64(one["v"]), P.f64(one["do"]), w.scale,
                                                   kv_len=kl, block_mask=bm)
        P.check_grad(P.f64(dq[b:b + 1, h:h + 1]), dq_r, f"padded block-sparse dQ ({b},{h})")
        P.check_grad(P.f64(dk[b:b + 1, h:h + 1]), dk_r, f"padded block-sparse dK ({b},{h})")
        P.check_grad(P.f64(dv[b:b + 1, h:h + 1]), dv_r, f"padded block-sparse dV ({b},{h})")


def _both_schedules(w, bm, window=None):
    """Forward and backward with the device mask alone and with its host
    copy; returns the two (o, lse, dq, dk, dv)."""
    g = P.to_gpu(make_inputs(w))
    out = []
    for m in (torch.from_numpy(bm).cuda(), fa.BlockMask(bm)):
        o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, window=window, block_mask=m)
        grads = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                            window=window, block_mask=m)
        out.append((o, lse) + tuple(grads))
    fa.fa_check()
    return out


def _agree(out):
    (o1, l1, dq1, dk1, dv1), (o2, l2, dq2, dk2, dv2) = out
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    diff = (dq1.float() - dq2.float()).abs().max().item()
    assert diff <= 2 ** -7 * dq1.float().abs().max().item(), diff


@pytest.mark.parametrize("d,Hkv", [(64, 8), (128, 2), (256, 8)])
def test_device_deal_with_skewed_costs(d, Hkv):
    """A mask with empty rows and columns (items of cost zero), a full row
    and a full column (the costliest items) and many ties: the device deal
    against the host plan (bit for bit, as above) and two heads against the
    oracle.  2 x 8 heads of 32 tiles are 512 items, four rounds of the deal
    on 152 SMs."""
    N = 4096
    T = N // 128
    bm = random_mask(T, 0.3, seed=d + Hkv)
    bm[[3, 17, 30]] = 0
    bm[:, [5, 21]] = 0
    bm[9] = 1
    bm[:, 12] = 1
    w = random_case(2, 8, N, d, seed=5 * d + Hkv, causal=False, h_kv=Hkv)
    out = _both_schedules(w, bm)
    _agree(out)
    o, lse, dq, dk, dv = out[0]
    inp = make_inputs(w)
    g = 8 // Hkv                            # query heads per K/V head
    for b, h in ((0, 1), (1, 8 - g)):
        kvh = h // g
        one = {"q": inp["q"][b:b + 1, h:h + 1], "do": inp["do"][b:b + 1, h:h + 1],
               "k": inp["k"][b:b + 1, kvh:kvh + 1], "v": inp["v"][b:b + 1, kvh:kvh + 1]}
        o_r, l_r = oracle.attention_fwd(P.f64(one["q"]), P.f64(one["k"]), P.f64(one["v"]),
                                        w.scale, block_mask=bm)
        P.check_o(P.f64(o[b:b + 1, h:h + 1]), o_r, f"device deal O ({b},{h})")
        P.check_lse(P.f64(lse[b:b + 1, h:h + 1]), l_r, f"device deal LSE ({b},{h})")
        dq_r, _, _, _ = oracle.attention_bwd(P.f64(one["q"]), P.f64(one["k"]), P.f64(one["v"]),
                                             P.f64(one["do"]), w.scale, block_mask=bm)
        P.check_grad(P.f64(dq[b:b + 1, h:h + 1]), dq_r, f"device deal dQ ({b},{h})")


@pytest.mark.parametrize("N", [257 * 128, 1025 * 128])
def test_device_deal_size_limits(N):
    """Past 256 tiles the forward's table does not fit its shared memory and
    the forward goes round-robin; past 1024 key blocks the backward's
    entries cannot hold them and the backward goes round-robin too.  Either
    way against the host plan, bit for bit (as above)."""
    from exact_attention_04_gb300.workloads import block_sparse_mask
    T = N // 128
    w = random_case(1, 2, N, 64, seed=T, causal=False)
    bm = block_sparse_mask(T, seed=T, band=1, n_random=2)
    _agree(_both_schedules(w, bm))
