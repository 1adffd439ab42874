"""The causal schedule covers every tile and every key block exactly once.

Plain causal attention runs on the paired schedule: tiles or key blocks
paired longest with shortest, round-robin, plus the host-planned tail of
single items. The same masks, given as a window (left unbounded, right 0)
with the causal flag off, run one item per unit round-robin. The arithmetic
of a tile, or of a key block, does not depend on the CTA that runs it or on
when it runs. So:
- the forward's O and LSE must agree bit for bit between the two schedules;
- so must the backward's dK and dV, which a key block accumulates in tensor
  memory;
- dQ is summed across key blocks in L2, in an order that differs from run
  to run, so it is compared within a few bf16 units.
A tile the schedule missed would leave its rows unwritten, and a key block
run twice would double its share of dQ. This test runs at the full headline
shapes, where the schedule has both paired units and a tail.
"""
import pytest
import torch

from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fabuild.build()
    fa.load()


def inputs(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    return w, {k: (None if t is None else t.cuda()) for k, t in inp.items()}


@pytest.mark.parametrize("name", ["large_head_b2_h16_n8192_d128_causal",
                                  "large_head_b2_h16_n8192_d256_causal",
                                  "gpt2_small_b8_h12_n1024_d64_causal"])
def test_forward_causal_schedule_matches_window_schedule(name):
    w, g = inputs(name)
    o1, lse1 = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=True)
    o2, lse2 = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=False, window=(-1, 0))
    fa.fa_check()
    assert torch.equal(o1, o2), (o1.float() - o2.float()).abs().max().item()
    assert torch.equal(lse1, lse2), (lse1 - lse2).abs().max().item()


@pytest.mark.parametrize("name", ["large_head_b2_h16_n8192_d128_causal",
                                  "large_head_b2_h16_n8192_d256_causal",
                                  "gpt2_small_b8_h12_n1024_d64_causal"])
def test_backward_causal_schedule_matches_window_schedule(name):
    w, g = inputs(name)
    o, lse = fa.forward(g["q"], g["k"], g["v"], scale=w.scale, causal=True)
    dq1, dk1, dv1 = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                                causal=True)
    dq2, dk2, dv2 = fa.backward(g["q"], g["k"], g["v"], o, lse, g["do"], scale=w.scale,
                                causal=False, window=(-1, 0))
    fa.fa_check()
    assert torch.equal(dk1, dk2), (dk1.float() - dk2.float()).abs().max().item()
    assert torch.equal(dv1, dv2), (dv1.float() - dv2.float()).abs().max().item()
    # fp32 sums in a different order, then rounded to bf16: at most one unit
    # in the last place (2^-7 of the value) where the order tipped the
    # rounding, which it does for few elements; a key block counted twice
    # would shift whole rows by about 1/64 of their size
    diff = (dq1.float() - dq2.float()).abs().max().item()
    assert diff <= 2 ** -7 * dq1.float().abs().max().item(), diff
    assert (dq1 != dq2).float().mean().item() < 0.01
