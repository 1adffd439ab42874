"""Python binding of libfa.so: argument marshalling only.

The functions named like the C ABI (``fa_fwd``, ``fa_bwd``, ...) take torch
tensors that already live on the GPU, check dtype / shape / contiguity, and
pass raw device pointers and the current CUDA stream to the library.  Every
step of the computation runs in the library's kernels; there is no fallback.
If libfa.so is missing or cannot be loaded the call raises.

``forward`` and ``backward`` are conveniences that allocate the outputs (and
the backward workspace) with torch before calling the C ABI.
"""
import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)

_lib = None


class FaVariant(ctypes.Structure):
    """fa_variant_t: K/V heads, flash-attn's (left, right) window (-1 =
    unbounded), a block mask (device pointer or None) and its host copy (host
    pointer or None)."""
    _fields_ = [("h_kv", ctypes.c_int), ("window_left", ctypes.c_int),
                ("window_right", ctypes.c_int), ("block_mask", ctypes.c_void_p),
                ("block_mask_host", ctypes.c_void_p)]


class BlockMask:
    """A block mask on the device together with its host copy.  Any function
    taking block_mask= accepts one in place of the CUDA tensor; the library
    then reads the host copy to balance its schedule (the results are the
    same either way)."""

    def __init__(self, mask, device=None):
        self.host = torch.as_tensor(mask).to(torch.uint8).cpu().contiguous()
        self.device = self.host.to("cuda" if device is None else device)


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)}")


def load():
    """Open libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m exact_attention_04_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, sz, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_prep.argtypes = [vp, vp, vp, i, i, i, i, vp, sz, vp]
        lib.fa_bwd_prep.restype = i
        lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, sz, vp]
        lib.fa_bwd_dkdv.restype = i
        lib.fa_bwd_dq.argtypes = [vp, i, i, i, i, f, vp, sz, vp]
        lib.fa_bwd_dq.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp,
                                       vp]
        lib.fa_bwd_noalloc.restype = i
        varp = ctypes.POINTER(FaVariant)
        lib.fa_fwd_v.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, varp, vp]
        lib.fa_fwd_v.restype = i
        lib.fa_bwd_v.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, varp,
                                 vp, sz, vp]
        lib.fa_bwd_v.restype = i
        lib.fa_bwd_dkdv_v.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, varp, vp, sz,
                                      vp]
        lib.fa_bwd_dkdv_v.restype = i
        lib.fa_decode_splits.argtypes = [i, i, i]
        lib.fa_decode_splits.restype = i
        lib.fa_decode_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.fa_decode_workspace_bytes.restype = sz
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, varp, i, vp, sz, vp]
        lib.fa_decode.restype = i
        fp = ctypes.POINTER(ctypes.c_float)
        lib.fa_fp8_quantize.argtypes = [vp, vp, vp, i, i, i, i, varp, vp, vp, vp, vp, vp, vp, vp]
        lib.fa_fp8_quantize.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, varp, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        lib.fa_selftest_wait_timeout.restype = i
        lib.fa_check.argtypes = [vp]
        lib.fa_check.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i
        _lib = lib
    return _lib


EXPORTS = ("fa_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_prep", "fa_bwd_dkdv",
           "fa_bwd_dq", "fa_bwd_noalloc", "fa_fwd_v", "fa_bwd_v", "fa_bwd_dkdv_v",
           "fa_decode_splits", "fa_decode_workspace_bytes", "fa_decode",
           "fa_fp8_quantize", "fa_fwd_fp8", "fa_selftest_wait_timeout", "fa_check",
           "fa_status_string", "fa_version")


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return load().fa_version()


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_qkv(name, t, shape=None):
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
        raise ValueError(f"{name}: expected a contiguous bf16 CUDA tensor [B,H,N,d]")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


def _check_kv_len(kv_len, B):
    if kv_len is None:
        return None
    if not kv_len.is_cuda or kv_len.dtype != torch.int32 or kv_len.numel() != B \
            or not kv_len.is_contiguous():
        raise ValueError("kv_len: expected a contiguous int32 CUDA tensor of length B")
    return kv_len


def _raise(status, where):
    if status != FA_OK:
        raise FAError(status, where)


def fa_fwd(q, k, v, o, lse, scale, causal=False, kv_len=None, stream=None):
    """Calls fa_fwd; q, k, v, o bf16 [B,H,N,d] and lse fp32 [B,H,N] on the GPU."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    _check_qkv("k", k, q.shape)
    _check_qkv("v", v, q.shape)
    _check_qkv("o", o, q.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N) \
            or not lse.is_contiguous():
        raise ValueError("lse: expected a contiguous fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    st = load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                       int(bool(causal)), _ptr(kv_len), _stream_ptr(stream))
    _raise(st, "fa_fwd")


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal=False, kv_len=None, workspace=None,
           stream=None):
    """Calls fa_bwd; workspace is a uint8 CUDA tensor of fa_bwd_workspace_bytes()."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse: expected fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    if workspace is None or not workspace.is_cuda:
        raise ValueError("workspace: expected a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    st = load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                       _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                       _ptr(kv_len), _ptr(workspace), nbytes, _stream_ptr(stream))
    _raise(st, "fa_bwd")


def _ws(workspace):
    if workspace is None or not workspace.is_cuda:
        raise ValueError("workspace: expected a CUDA tensor")
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def fa_bwd_prep(o, do, lse, workspace, stream=None):
    """First backward phase: D, LSE*log2(e) into the workspace; zero the dQ accumulator."""
    _check_qkv("o", o)
    B, H, N, d = o.shape
    _check_qkv("do", do, o.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse: expected fp32 CUDA tensor [B,H,N]")
    wp, wn = _ws(workspace)
    _raise(load().fa_bwd_prep(_ptr(o), _ptr(do), _ptr(lse), B, H, N, d, wp, wn,
                              _stream_ptr(stream)), "fa_bwd_prep")


def fa_bwd_dkdv(q, k, v, do, dk, dv, scale, causal=False, kv_len=None, workspace=None,
                stream=None):
    """Second backward phase: dK, dV and the fp32 dQ accumulation."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("do", do), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    kv_len = _check_kv_len(kv_len, B)
    wp, wn = _ws(workspace)
    _raise(load().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), B, H, N,
                              d, float(scale), int(bool(causal)), _ptr(kv_len), wp, wn,
                              _stream_ptr(stream)), "fa_bwd_dkdv")


def fa_bwd_dq(dq, scale, workspace, stream=None):
    """Third backward phase: dQ = bf16(scale * accumulator)."""
    _check_qkv("dq", dq)
    B, H, N, d = dq.shape
    wp, wn = _ws(workspace)
    _raise(load().fa_bwd_dq(_ptr(dq), B, H, N, d, float(scale), wp, wn, _stream_ptr(stream)),
           "fa_bwd_dq")


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, scale, causal=False, kv_len=None,
                   stream=None):
    """fa_bwd without a workspace, for callers that cannot allocate device
    memory: the library's own fixed scratch array is used instead (see
    include/fa.h for its size limit and the rule that overlapping calls race)."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse: expected fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    _raise(load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                 int(bool(causal)), _ptr(kv_len), _stream_ptr(stream)),
           "fa_bwd_noalloc")


def _check_block_mask(bm, N):
    """(device pointer, host pointer) of a block mask: a contiguous uint8
    CUDA tensor [T, T], T = ceil(N/128), or a BlockMask holding one and its
    host copy.  The caller keeps bm alive across the call."""
    if bm is None:
        return None, None
    t = -(-N // 128)
    host = None
    if isinstance(bm, BlockMask):
        host, bm = bm.host, bm.device
        if host.dtype != torch.uint8 or tuple(host.shape) != (t, t) or not host.is_contiguous():
            raise ValueError(f"block_mask: expected a host copy of shape [{t}, {t}]")
    if bm.dtype != torch.uint8 or not bm.is_cuda or tuple(bm.shape) != (t, t) \
            or not bm.is_contiguous():
        raise ValueError(f"block_mask: expected a contiguous uint8 CUDA tensor [{t}, {t}]")
    return bm.data_ptr(), None if host is None else host.data_ptr()


def _variant(q, k, window, block_mask=None):
    """fa_variant_t for K/V of k's head count, the (left, right) window and a
    block mask."""
    B, H, N, d = q.shape
    if k.dim() != 4 or (k.shape[0], k.shape[2], k.shape[3]) != (B, N, d) or k.shape[1] < 1 \
            or H % k.shape[1]:
        raise ValueError(f"k: shape {tuple(k.shape)} does not group the {H} query heads")
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    return FaVariant(int(k.shape[1]), wl, wr, *_check_block_mask(block_mask, N))


def fa_fwd_v(q, k, v, o, lse, scale, causal=False, kv_len=None, window=None, stream=None,
             block_mask=None):
    """Calls fa_fwd_v: k, v are [B,H_kv,N,d] (H_kv divides H); window is
    flash-attn's (left, right), -1 = unbounded; block_mask a uint8 CUDA
    tensor [ceil(N/128)]^2, zero where a (query block, key block) is skipped,
    or a BlockMask (the same with its host copy, for a balanced schedule)."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    var = _variant(q, k, window, block_mask)
    _check_qkv("k", k, k.shape)
    _check_qkv("v", v, k.shape)
    _check_qkv("o", o, q.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N) \
            or not lse.is_contiguous():
        raise ValueError("lse: expected a contiguous fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    st = load().fa_fwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                         int(bool(causal)), _ptr(kv_len), ctypes.byref(var), _stream_ptr(stream))
    _raise(st, "fa_fwd_v")


def fa_bwd_v(q, k, v, o, do, lse, dq, dk, dv, scale, causal=False, kv_len=None, window=None,
             workspace=None, stream=None, block_mask=None):
    """Calls fa_bwd_v: k, v, dk, dv are [B,H_kv,N,d]; dk, dv sum over each group."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    var = _variant(q, k, window, block_mask)
    for name, t in (("o", o), ("do", do), ("dq", dq)):
        _check_qkv(name, t, q.shape)
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, k.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse: expected fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    wp, wn = _ws(workspace)
    st = load().fa_bwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                         _ptr(kv_len), ctypes.byref(var), wp, wn, _stream_ptr(stream))
    _raise(st, "fa_bwd_v")


def fa_bwd_dkdv_v(q, k, v, do, dk, dv, scale, causal=False, kv_len=None, window=None,
                  workspace=None, stream=None, block_mask=None):
    """Second backward phase for a variant: k, v, dk, dv are [B,H_kv,N,d]."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    var = _variant(q, k, window, block_mask)
    _check_qkv("do", do, q.shape)
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, k.shape)
    kv_len = _check_kv_len(kv_len, B)
    wp, wn = _ws(workspace)
    _raise(load().fa_bwd_dkdv_v(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), B, H,
                                N, d, float(scale), int(bool(causal)), _ptr(kv_len),
                                ctypes.byref(var), wp, wn, _stream_ptr(stream)), "fa_bwd_dkdv_v")


def fa_decode_splits(B, h_kv, Nk) -> int:
    return int(load().fa_decode_splits(B, h_kv, Nk))


def fa_decode_workspace_bytes(B, H, Nq, d, splits) -> int:
    return int(load().fa_decode_workspace_bytes(B, H, Nq, d, splits))


def fa_decode(q, k, v, o, lse, scale, causal=False, kv_len=None, window=None, splits=1,
              workspace=None, stream=None):
    """Calls fa_decode: q, o [B,H,Nq,d]; k, v [B,H_kv,Nk,d] (H_kv divides H);
    lse fp32 [B,H,Nq]; workspace of fa_decode_workspace_bytes()."""
    _check_qkv("q", q)
    B, H, Nq, d = q.shape
    _check_qkv("k", k)
    Hkv, Nk = k.shape[1], k.shape[2]
    if (k.shape[0], k.shape[3]) != (B, d) or Hkv < 1 or H % Hkv:
        raise ValueError(f"k: shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    _check_qkv("v", v, k.shape)
    _check_qkv("o", o, q.shape)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, Nq) \
            or not lse.is_contiguous():
        raise ValueError("lse: expected a contiguous fp32 CUDA tensor [B,H,Nq]")
    kv_len = _check_kv_len(kv_len, B)
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    var = FaVariant(int(Hkv), wl, wr)
    wp, wn = _ws(workspace)
    _raise(load().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                            float(scale), int(bool(causal)), _ptr(kv_len), ctypes.byref(var),
                            int(splits), wp, wn, _stream_ptr(stream)), "fa_decode")


def decode(q, k, v, scale=None, causal=False, kv_len=None, window=None, splits=None,
           stream=None):
    """(O, LSE) of split-KV decoding with outputs and workspace allocated by
    torch; splits defaults to the library's choice for this GPU."""
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if splits is None:
        splits = max(1, fa_decode_splits(B, Hkv, Nk))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws = torch.empty(fa_decode_workspace_bytes(B, H, Nq, d, splits), dtype=torch.uint8,
                     device=q.device)
    fa_decode(q, k, v, o, lse, default_scale(d) if scale is None else scale, causal, kv_len,
              window, splits, ws, stream)
    return o, lse


def fp8_buffers(B, H, Hkv, N, d, device):
    """Empty E4M3 buffers and scales in the layouts fa_fp8_quantize writes."""
    nb = -(-N // 128)
    u8 = dict(dtype=torch.uint8, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return {"q8": torch.empty(B, H, N, d, **u8), "q_scale": torch.empty(B, H, nb, **f32),
            "k8": torch.empty(B, Hkv, N, d, **u8), "k_scale": torch.empty(B, Hkv, nb, **f32),
            "v8t": torch.zeros(B, Hkv, d, nb * 128, **u8), "v_scale": torch.empty(B, Hkv, **f32)}


def fa_fp8_quantize(q, k, v, buf, stream=None):
    """Calls fa_fp8_quantize into buf (from fp8_buffers)."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    var = _variant(q, k, None)
    _check_qkv("k", k, k.shape)
    _check_qkv("v", v, k.shape)
    _raise(load().fa_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, ctypes.byref(var),
                                  _ptr(buf["q8"]), _ptr(buf["q_scale"]), _ptr(buf["k8"]),
                                  _ptr(buf["k_scale"]), _ptr(buf["v8t"]), _ptr(buf["v_scale"]),
                                  _stream_ptr(stream)), "fa_fp8_quantize")


def fa_fwd_fp8(buf, o, lse, scale, causal=False, kv_len=None, window=None, stream=None,
               block_mask=None):
    """Calls fa_fwd_fp8 on E4M3 buffers (from fp8_buffers / fa_fp8_quantize)."""
    B, H, N, d = buf["q8"].shape
    Hkv = buf["k8"].shape[1]
    _check_qkv("o", o, (B, H, N, d))
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse: expected fp32 CUDA tensor [B,H,N]")
    kv_len = _check_kv_len(kv_len, B)
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    var = FaVariant(int(Hkv), wl, wr, *_check_block_mask(block_mask, N))
    _raise(load().fa_fwd_fp8(_ptr(buf["q8"]), _ptr(buf["q_scale"]), _ptr(buf["k8"]),
                             _ptr(buf["k_scale"]), _ptr(buf["v8t"]), _ptr(buf["v_scale"]),
                             _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(bool(causal)),
                             _ptr(kv_len), ctypes.byref(var), _stream_ptr(stream)), "fa_fwd_fp8")


def forward_fp8(q, k, v, scale=None, causal=False, kv_len=None, window=None, stream=None,
                block_mask=None):
    """(O, LSE, E4M3 buffers): quantise bf16 Q, K, V and run the FP8 forward."""
    B, H, N, d = q.shape
    buf = fp8_buffers(B, H, k.shape[1], N, d, q.device)
    fa_fp8_quantize(q, k, v, buf, stream)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_fp8(buf, o, lse, default_scale(d) if scale is None else scale, causal, kv_len, window,
               stream, block_mask)
    return o, lse, buf


def fa_selftest_wait_timeout(timeout_us, stream=None):
    """Enqueues the bounded-wait self-test (see include/fa.h); the next
    fa_check() must raise FAError with FA_ERR_TIMEOUT."""
    _raise(load().fa_selftest_wait_timeout(int(timeout_us), _stream_ptr(stream)),
           "fa_selftest_wait_timeout")


def fa_check(stream=None):
    """Waits for the stream; raises FAError if a kernel timed out or failed."""
    _raise(load().fa_check(_stream_ptr(stream)), "fa_check")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def forward(q, k, v, scale=None, causal=False, kv_len=None, window=None, stream=None,
            block_mask=None):
    """(O, LSE) with outputs allocated by torch on q's device.  K/V with fewer
    heads than Q, a window or a block mask go through fa_fwd_v."""
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    sc = default_scale(d) if scale is None else scale
    if window is None and block_mask is None and k.shape == q.shape:
        fa_fwd(q, k, v, o, lse, sc, causal, kv_len, stream)
    else:
        fa_fwd_v(q, k, v, o, lse, sc, causal, kv_len, window, stream, block_mask)
    return o, lse


def workspace(B, H, N, d, device):
    return torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)


def backward(q, k, v, o, lse, do, scale=None, causal=False, kv_len=None, ws=None, window=None,
             stream=None, block_mask=None):
    """(dQ, dK, dV) with outputs (and, if not given, the workspace) allocated by
    torch; dK, dV are shaped like k."""
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    if ws is None:
        ws = workspace(B, H, N, d, q.device)
    sc = default_scale(d) if scale is None else scale
    if window is None and block_mask is None and k.shape == q.shape:
        fa_bwd(q, k, v, o, do, lse, dq, dk, dv, sc, causal, kv_len, ws, stream)
    else:
        fa_bwd_v(q, k, v, o, do, lse, dq, dk, dv, sc, causal, kv_len, window, ws, stream,
                 block_mask)
    return dq, dk, dv
