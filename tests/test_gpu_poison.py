"""Every output element written, nothing written outside the outputs.

Each output lives inside a larger buffer filled with NaN (bf16 / fp32) or
0xFF bytes (E4M3 NaN codes), with 256 bytes of guard on either side.  After
the call the output must hold no NaN (rows that see no key hold 0 and an LSE
of -inf) and every guard byte must be as it was.  Workspaces are filled with
0xFF too, since their contents on entry must not matter.  Small ragged shapes
put partial tiles and key blocks at the edges of the buffers.
"""
import pytest
import torch

from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import block_sparse_mask, make_inputs, random_case

pytestmark = pytest.mark.gpu

GUARD_BYTES = 256


class Guarded:
    """A tensor of `shape` inside a buffer poisoned with `fill`."""

    def __init__(self, shape, dtype, fill):
        n = 1
        for s in shape:
            n *= s
        self.g = GUARD_BYTES // torch.tensor([], dtype=dtype).element_size()
        self.n = n
        self.buf = torch.full((n + 2 * self.g,), fill, dtype=dtype, device="cuda")
        self.t = self.buf[self.g:self.g + n].view(shape)

    def guards_intact(self, fill):
        head, tail = self.buf[:self.g], self.buf[self.g + self.n:]
        if isinstance(fill, float) and fill != fill:     # NaN
            return bool(torch.isnan(head.float()).all() and torch.isnan(tail.float()).all())
        return bool((head == fill).all() and (tail == fill).all())


NAN = float("nan")


def _outputs(B, H, N, d):
    return Guarded((B, H, N, d), torch.bfloat16, NAN), Guarded((B, H, N), torch.float32, NAN)


def _assert_written(*gs):
    for g in gs:
        assert g.guards_intact(NAN), "a kernel wrote outside its output"
        assert not torch.isnan(g.t.float()).any(), "an output element was not written"


def _poisoned_workspace(nbytes):
    return torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")


FWD_CASES = [
    # B, H, N, d, causal, kv_len range
    (2, 3, 129, 64, True, (1, 129)),
    (3, 2, 383, 128, False, (0, 383)),     # kv_len 0: rows that see no key
    (1, 3, 17, 256, True, None),
    (2, 2, 257, 128, False, (100, 257)),
    (1, 2, 640, 64, False, None),
]


@pytest.mark.parametrize("B,H,N,d,causal,kv", FWD_CASES)
def test_forward_and_backward_write_exactly_their_outputs(B, H, N, d, causal, kv):
    w = random_case(B, H, N, d, seed=N + d, causal=causal, kv_len_range=kv)
    inp = make_inputs(w)
    if kv is not None and kv[0] == 0:
        inp["kv_len"][0] = 0
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    o, lse = _outputs(B, H, N, d)
    fa.fa_fwd(g["q"], g["k"], g["v"], o.t, lse.t, w.scale, causal, g["kv_len"])
    fa.fa_check()
    _assert_written(o, lse)
    dq, dk, dv = (Guarded((B, H, N, d), torch.bfloat16, NAN) for _ in range(3))
    ws = _poisoned_workspace(fa.fa_bwd_workspace_bytes(B, H, N, d))
    fa.fa_bwd(g["q"], g["k"], g["v"], o.t, g["do"], lse.t, dq.t, dk.t, dv.t, w.scale, causal,
              g["kv_len"], workspace=ws)
    fa.fa_check()
    _assert_written(dq, dk, dv)
    ref = fa.backward(g["q"], g["k"], g["v"], o.t, lse.t, g["do"], scale=w.scale, causal=causal,
                      kv_len=g["kv_len"])
    fa.fa_check()
    # the poisoned workspace gives the same dK, dV as a fresh one
    assert torch.equal(dk.t, ref[1]) and torch.equal(dv.t, ref[2])


@pytest.mark.parametrize("d", [64, 128])
def test_variants_write_exactly_their_outputs(d):
    """GQA with a two-sided window, and a block mask, forward and backward."""
    B, H, Hkv, N = 2, 4, 2, 300
    w = random_case(B, H, N, d, seed=7 * d, causal=False, h_kv=Hkv, window=(90, 40))
    g = {k: (None if t is None else t.cuda()) for k, t in make_inputs(w).items()}
    for window, bm in (((90, 40), None),
                       (None, torch.from_numpy(block_sparse_mask(3, seed=1, band=0, n_global=1,
                                                                 n_random=1)).cuda())):
        o, lse = _outputs(B, H, N, d)
        fa.fa_fwd_v(g["q"], g["k"], g["v"], o.t, lse.t, w.scale, kv_len=g["kv_len"],
                    window=window, block_mask=bm)
        fa.fa_check()
        _assert_written(o, lse)
        dq = Guarded((B, H, N, d), torch.bfloat16, NAN)
        dk, dv = (Guarded((B, Hkv, N, d), torch.bfloat16, NAN) for _ in range(2))
        ws = _poisoned_workspace(fa.fa_bwd_workspace_bytes(B, H, N, d))
        fa.fa_bwd_v(g["q"], g["k"], g["v"], o.t, g["do"], lse.t, dq.t, dk.t, dv.t, w.scale,
                    kv_len=g["kv_len"], window=window, workspace=ws, block_mask=bm)
        fa.fa_check()
        _assert_written(dq, dk, dv)


def test_decode_writes_exactly_its_outputs():
    B, H, Hkv, Nq, Nk, d = 3, 4, 2, 2, 1000, 128
    gen = torch.Generator().manual_seed(11)
    q = torch.randn(B, H, Nq, d, generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn(B, Hkv, Nk, d, generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, Nk, d, generator=gen).to(torch.bfloat16).cuda()
    kv_len = torch.tensor([1000, 1, 0], dtype=torch.int32, device="cuda")
    for splits in (1, 3):
        o, lse = _outputs(B, H, Nq, d)
        ws = _poisoned_workspace(fa.fa_decode_workspace_bytes(B, H, Nq, d, splits))
        fa.fa_decode(q, k, v, o.t, lse.t, d ** -0.5, causal=True, kv_len=kv_len, splits=splits,
                     workspace=ws)
        fa.fa_check()
        _assert_written(o, lse)


def test_fp8_quantiser_and_forward_write_exactly_their_outputs():
    B, H, Hkv, N, d = 2, 4, 2, 200, 128
    w = random_case(B, H, N, d, seed=13, causal=True, h_kv=Hkv, kv_len_range=(1, 200))
    g = {k: (None if t is None else t.cuda()) for k, t in make_inputs(w, with_grad_out=False).items()}
    nb = -(-N // 128)
    u8, f32 = torch.uint8, torch.float32
    gb = {"q8": Guarded((B, H, N, d), u8, 0xFF), "q_scale": Guarded((B, H, nb), f32, NAN),
          "k8": Guarded((B, Hkv, N, d), u8, 0xFF), "k_scale": Guarded((B, Hkv, nb), f32, NAN),
          "v8t": Guarded((B, Hkv, d, nb * 128), u8, 0xFF), "v_scale": Guarded((B, Hkv), f32, NAN)}
    buf = {k: x.t for k, x in gb.items()}
    fa.fa_fp8_quantize(g["q"], g["k"], g["v"], buf)
    fa.fa_check()
    for name, x in gb.items():
        if x.t.dtype == torch.uint8:
            assert x.guards_intact(0xFF), name
            # 0x7F and 0xFF are E4M3's NaN codes: none may remain
            assert not ((x.t & 0x7F) == 0x7F).any(), name
        else:
            _assert_written(x)
    o, lse = _outputs(B, H, N, d)
    fa.fa_fwd_fp8(buf, o.t, lse.t, w.scale, causal=True, kv_len=g["kv_len"])
    fa.fa_check()
    _assert_written(o, lse)
