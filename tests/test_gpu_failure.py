"""Failure detection without a GPU fault: a kernel whose wait is never
satisfied gives up at its limit, records FA_ERR_TIMEOUT in the device status
word and returns; the host reads it through fa_check, the word is cleared,
and the context keeps working."""
import pytest
import torch

from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa
from exact_attention_04_gb300.workloads import make_inputs, random_case

import parity as P
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fabuild.build()
    fa.load()


def test_wait_that_never_completes_reports_timeout_and_device_stays_usable():
    fa.fa_check()                                  # start from a clean status word
    fa.fa_selftest_wait_timeout(3000)              # 3 ms limit
    with pytest.raises(fa.FAError) as e:
        fa.fa_check()
    assert e.value.status == fa.FA_ERR_TIMEOUT
    fa.fa_check()                                  # the word was cleared
    w = random_case(1, 2, 300, 64, seed=12, causal=True)
    inp = make_inputs(w)
    g, o, lse = P.gpu_forward(w, inp)
    o_ref, lse_ref = oracle.attention_fwd(P.f64(inp["q"]), P.f64(inp["k"]), P.f64(inp["v"]),
                                          w.scale, causal=True)
    P.check_o(P.f64(o), o_ref, "after timeout O")
    P.check_lse(P.f64(lse), lse_ref, "after timeout LSE")
