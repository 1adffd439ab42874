"""Host-side checks of the C-ABI library (no GPU needed).

The library must load, export every function include/fa.h declares, and
reject bad arguments with the documented status codes before touching the
device.
"""
import ctypes
import os
import re

import pytest

from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_check",
                     "fa_status_string", "fa_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(fa.EXPORTS)


def test_status_strings_and_version(lib):
    assert fa.fa_status_string(fa.FA_OK) == "FA_OK"
    assert fa.fa_status_string(fa.FA_ERR_TIMEOUT) == "FA_ERR_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"
    assert fa.fa_version() >= 10200         # fa_variant_t with block_mask_host


def test_variant_layout_matches_the_header(tmp_path):
    """The binding's FaVariant has the size and member offsets that a C
    compiler gives fa_variant_t from include/fa.h."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "fa.h"\n'
        "int main(void) { printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(fa_variant_t),"
        " offsetof(fa_variant_t, h_kv), offsetof(fa_variant_t, window_left),"
        " offsetof(fa_variant_t, window_right), offsetof(fa_variant_t, block_mask),"
        " offsetof(fa_variant_t, block_mask_host)); return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    V = fa.FaVariant
    assert got == [ctypes.sizeof(V), V.h_kv.offset, V.window_left.offset,
                   V.window_right.offset, V.block_mask.offset, V.block_mask_host.offset]


def test_workspace_bytes(lib):
    B, H, N, d = 2, 3, 200, 64
    npad = 256
    stat = -(-B * H * npad * 4 // 256) * 256
    acc = -(-B * H * npad * d * 4 // 256) * 256
    order = -(-(npad // 128) * 4 // 256) * 256     # the key blocks' cost-sorted order
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) == 2 * stat + acc + order
    assert fa.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 96) == 0


P = ctypes.c_void_p


def fwd(lib, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=1, N=128, d=64,
        scale=0.125, causal=0, kv=None):
    return lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, causal,
                      P(kv) if kv else None, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, q=0) == fa.FA_ERR_INVALID_ARG             # null pointer
    assert fwd(lib, o=0x1008) == fa.FA_ERR_INVALID_ARG        # misaligned output
    assert fwd(lib, lse=0x1002) == fa.FA_ERR_INVALID_ARG      # misaligned lse
    assert fwd(lib, kv=0x1001) == fa.FA_ERR_INVALID_ARG       # misaligned kv_len
    assert fwd(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, B=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=32) == fa.FA_ERR_UNSUPPORTED
    assert fwd(lib, B=1 << 14, H=1 << 10, N=1 << 10, d=64) == fa.FA_ERR_INVALID_ARG  # 2^31 elements


def test_backward_argument_errors(lib):
    ok = 0x1000

    def bwd(ws=ok, ws_bytes=1 << 40, d=64, dq=ok, scale=0.125):
        return lib.fa_bwd(P(ok), P(ok), P(ok), P(ok), P(ok), P(ok), P(dq), P(ok), P(ok), 1, 1, 128,
                          d, scale, 0, None, P(ws), ws_bytes, None)
    assert bwd(dq=0) == fa.FA_ERR_INVALID_ARG
    assert bwd(ws=0) == fa.FA_ERR_INVALID_ARG
    assert bwd(ws=0x1010) == fa.FA_ERR_INVALID_ARG            # workspace must be 256-aligned
    assert bwd(ws_bytes=16) == fa.FA_ERR_INVALID_ARG          # too small
    assert bwd(d=80) == fa.FA_ERR_UNSUPPORTED
    assert bwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 128)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q, lse, 0.125)


def test_variant_argument_errors(lib):
    """fa_fwd_v / fa_bwd_v reject a K/V head count that does not divide H and
    window sides below -1 before touching the device."""
    ok = 0x1000

    def fwd_v(h_kv, wl=-1, wr=-1, H=4):
        var = fa.FaVariant(h_kv, wl, wr)
        return lib.fa_fwd_v(P(ok), P(ok), P(ok), P(ok), P(ok), 1, H, 128, 64, 0.125, 0, None,
                            ctypes.byref(var), None)

    def bwd_v(h_kv, wl=-1, wr=-1, H=4):
        var = fa.FaVariant(h_kv, wl, wr)
        return lib.fa_bwd_v(P(ok), P(ok), P(ok), P(ok), P(ok), P(ok), P(ok), P(ok), P(ok), 1, H,
                            128, 64, 0.125, 0, None, ctypes.byref(var), P(ok), 1 << 40, None)
    for call in (fwd_v, bwd_v):
        assert call(3) == fa.FA_ERR_INVALID_ARG          # 3 does not divide 4
        assert call(0) == fa.FA_ERR_INVALID_ARG
        assert call(8) == fa.FA_ERR_INVALID_ARG          # more K/V heads than query heads
        assert call(2, wl=-2) == fa.FA_ERR_INVALID_ARG
        assert call(2, wr=-5) == fa.FA_ERR_INVALID_ARG


def test_block_mask_binding_passes_both_copies(lib):
    """A BlockMask gives the variant its device pointer and its host copy's
    pointer; a plain tensor gives no host copy; wrong shapes are refused."""
    import torch

    class FakeCuda:                      # a stand-in for a CUDA uint8 tensor (no GPU here)
        dtype, is_cuda, shape = torch.uint8, True, (2, 2)

        def is_contiguous(self):
            return True

        def data_ptr(self):
            return 0x1000

    bm = fa.BlockMask.__new__(fa.BlockMask)
    bm.host = torch.tensor([[1, 0], [1, 1]], dtype=torch.uint8)
    bm.device = FakeCuda()
    assert fa._check_block_mask(bm, 256) == (0x1000, bm.host.data_ptr())
    assert fa._check_block_mask(FakeCuda(), 200) == (0x1000, None)
    assert fa._check_block_mask(None, 200) == (None, None)
    with pytest.raises(ValueError):
        fa._check_block_mask(bm, 512)     # T = 4, not 2
    bm.host = torch.ones(2, 3, dtype=torch.uint8)
    with pytest.raises(ValueError):
        fa._check_block_mask(bm, 256)


def test_variant_binding_checks_shapes(lib):
    import torch
    q = torch.zeros(1, 4, 128, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 3, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa._variant(q, k, None)


def test_selftest_rejects_limits_out_of_range(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(2000000, None) == fa.FA_ERR_INVALID_ARG


def test_fp8_argument_errors(lib):
    """fa_fp8_quantize / fa_fwd_fp8: null or misaligned buffers, d = 64 (no
    E4M3 kernel) and bad K/V head counts are refused before the device."""
    ok = 0x1000

    def quant(q8=ok, qs=ok, d=128, h_kv=1, H=2):
        var = fa.FaVariant(h_kv, -1, -1)
        return lib.fa_fp8_quantize(P(ok), P(ok), P(ok), 1, H, 128, d, ctypes.byref(var), P(q8),
                                   P(qs), P(ok), P(ok), P(ok), P(ok), None)

    def fwd8(v8t=ok, lse=ok, d=128, N=128, scale=0.125, h_kv=1, H=2):
        var = fa.FaVariant(h_kv, -1, -1)
        return lib.fa_fwd_fp8(P(ok), P(ok), P(ok), P(ok), P(v8t), P(ok), P(ok), P(lse), 1, H, N,
                              d, scale, 1, None, ctypes.byref(var), None)
    assert quant(q8=0) == fa.FA_ERR_INVALID_ARG
    assert quant(q8=0x1008) == fa.FA_ERR_INVALID_ARG       # codes must be 16-byte aligned
    assert quant(qs=0x1002) == fa.FA_ERR_INVALID_ARG       # scales must be 4-byte aligned
    assert quant(d=64) == fa.FA_ERR_UNSUPPORTED
    assert quant(h_kv=3) == fa.FA_ERR_INVALID_ARG
    assert fwd8(v8t=0) == fa.FA_ERR_INVALID_ARG
    assert fwd8(lse=0x1001) == fa.FA_ERR_INVALID_ARG
    assert fwd8(d=64) == fa.FA_ERR_UNSUPPORTED
    assert fwd8(d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd8(N=0) == fa.FA_ERR_INVALID_ARG
    assert fwd8(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd8(h_kv=4) == fa.FA_ERR_INVALID_ARG


def test_decode_refuses_a_block_mask(lib):
    """fa_decode has no block-sparse schedule: a variant with a block mask is
    refused before the device (the mask pointer is never read)."""
    ok = 0x1000
    var = fa.FaVariant(2, -1, -1, 0x2000)
    st = lib.fa_decode(P(ok), P(ok), P(ok), P(ok), P(ok), 1, 2, 1, 256, 128, 0.1, 1, None,
                       ctypes.byref(var), 1, P(0x100000), 1 << 20, None)
    assert st == fa.FA_ERR_UNSUPPORTED


def test_decode_split_choice(lib):
    """fa_decode_splits: with fewer K/V heads than SMs, the most chunks of at
    least 8 key blocks that fit one wave; always within [1, key blocks]."""
    import torch
    sms = (torch.cuda.get_device_properties(0).multi_processor_count
           if torch.cuda.is_available() else 148)
    assert fa.fa_decode_splits(4, 8, 32768) == min(sms // 32, 256 // 8)
    assert fa.fa_decode_splits(1, 1, 1000) == 1                  # 8 blocks: one chunk
    assert fa.fa_decode_splits(1, 2, 131072) == min(sms // 2, 1024 // 8)
    for B, hk, nk in ((64, 8, 4096), (3, 100, 20000), (1, 1, 1), (2, 40, 128 * 64)):
        s = fa.fa_decode_splits(B, hk, nk)
        assert 1 <= s <= -(-nk // 128)
        if B * hk < sms:
            assert B * hk * s <= sms
    assert fa.fa_decode_splits(0, 8, 100) == 0


def test_noalloc_backward_reports_fa_bwd_status_codes(lib):
    """fa_bwd_noalloc checks its arguments as fa_bwd does, in the same order,
    so a bad call gets the same status from both (here every case fails
    before the device is touched, or at the device lookup on a host without
    a GPU).  Only a problem larger than the fixed scratch differs: it is
    refused with FA_ERR_INVALID_ARG, as fa_bwd refuses a workspace too small."""
    import torch
    ok = 0x1000

    def both(q=ok, lse=ok, kv=None, B=1, H=1, N=128, d=64, scale=0.125):
        a = lib.fa_bwd(P(q), P(ok), P(ok), P(ok), P(ok), P(lse), P(ok), P(ok), P(ok), B, H, N,
                       d, scale, 0, P(kv) if kv else None, P(0x100000), 1 << 40, None)
        b = lib.fa_bwd_noalloc(P(q), P(ok), P(ok), P(ok), P(ok), P(lse), P(ok), P(ok), P(ok),
                               B, H, N, d, scale, 0, P(kv) if kv else None, None)
        return a, b
    cases = [dict(q=0), dict(q=0x1008), dict(lse=0x1002), dict(kv=0x1001), dict(B=0),
             dict(B=0, d=100), dict(N=0, d=32), dict(d=100), dict(d=100, scale=0.0),
             dict(scale=float("nan")), dict(B=1 << 14, H=1 << 10, N=1 << 10)]
    if not torch.cuda.is_available():
        cases.append({})                 # valid arguments: both stop at the device lookup
    for c in cases:
        a, b = both(**c)
        assert a == b, (c, a, b)
        assert a != fa.FA_OK
    assert both(B=1, H=1, N=131072, d=128)[1] == fa.FA_ERR_INVALID_ARG
