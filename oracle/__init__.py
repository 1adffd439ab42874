"""CPU fp64 oracle for exact attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
library under ``exact_attention_04_gb300`` never imports it, and this package
imports nothing from that library: the two share only the seeded input
generators, which hold none of the method's arithmetic.

Two parts:

* ``attn_oracle.c`` (loaded here through ctypes): the plain definition of
  attention forward and backward, written out row by row in double precision.
  See the header of that file for the passages it follows.
* ``softmax_ref.py``: the pages' softmax recurrences (three-pass safe softmax,
  the online normaliser, the one-pass softmax-times-V and the associative
  block merge) in numpy float64, and a tiled forward built from them.

Every input is float64; callers widen bf16 tensors exactly before calling.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.fa_oracle_forward_v.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_int,
                                            c_double, c_int, ip, c_int, c_int, c_int]
        lib.fa_oracle_forward_v.restype = c_int
        u8p = ctypes.POINTER(ctypes.c_ubyte)
        lib.fa_oracle_forward_m.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_int,
                                            c_double, c_int, ip, c_int, c_int, u8p, c_int, c_int]
        lib.fa_oracle_forward_m.restype = c_int
        lib.fa_oracle_backward_m.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int,
                                             c_int, c_int, c_double, c_int, ip, c_int, c_int,
                                             u8p, c_int, c_int]
        lib.fa_oracle_backward_m.restype = c_int
        lib.fa_oracle_forward_rows_v.argtypes = [dp, dp, dp, c_int, c_int, c_double, c_int, c_int,
                                                 c_int, c_int, ip, c_int, dp, dp, c_int]
        lib.fa_oracle_forward_rows_v.restype = c_int
        lib.fa_oracle_backward_v.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int,
                                             c_int, c_int, c_double, c_int, ip, c_int, c_int, c_int]
        lib.fa_oracle_backward_v.restype = c_int
        lib.fa_oracle_decode.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_double, c_int, ip, c_int, c_int, c_int]
        lib.fa_oracle_decode.restype = c_int
        lib.fa_oracle_num_threads.argtypes = []
        lib.fa_oracle_num_threads.restype = c_int
        _lib = lib
    return _lib


def _f64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _ptr(a, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    """Threads the oracle uses by default: every host core."""
    return max(1, os.cpu_count() or 1)


def compiled_threads() -> int:
    """OpenMP's own thread limit inside the library (1 when built without OpenMP)."""
    return _load().fa_oracle_num_threads()


def _kv(kv_len, B):
    if kv_len is None:
        return None, None
    kv = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32).reshape(B))
    return kv, _ptr(kv, ctypes.c_int)


def _window(window):
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if wl < -1 or wr < -1:
        raise ValueError("window sides are -1 (unbounded) or >= 0")
    return wl, wr


def _block_mask(block_mask, N, block):
    """(array, pointer) of a block mask: a [ceil(N/block), ceil(N/block)]
    array, nonzero where a (query block, key block) pair is computed."""
    if block_mask is None:
        return None, None
    if block < 1:
        raise ValueError("block size must be positive")
    t = -(-N // block)
    bm = np.ascontiguousarray((np.asarray(block_mask) != 0).astype(np.uint8))
    if bm.shape != (t, t):
        raise ValueError(f"block mask must be [{t}, {t}] for N={N}, block {block}")
    return bm, _ptr(bm, ctypes.c_ubyte)


def _heads(q, k):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or Hkv < 1 or H % Hkv:
        raise ValueError(f"K/V shape {k.shape} does not group the {H} query heads")
    return B, H, Hkv, N, d


def attention_fwd(q, k, v, scale, causal=False, kv_len=None, threads=None, window=None,
                  block_mask=None, block=128):
    """O [B,H,N,d] and LSE [B,H,N] of exact attention (float64 numpy arrays).

    k, v are [B,H_kv,N,d] with H_kv dividing H (query head h reads K/V head
    h // (H // H_kv)); window is flash-attn's (left, right), -1 = unbounded;
    block_mask, [ceil(N/block)]^2, hides the keys of every (query block, key
    block) pair where it is zero, for every head."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, d = _heads(q, k)
    assert v.shape == k.shape
    wl, wr = _window(window)
    bm, bmp = _block_mask(block_mask, N, block)
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    kv, kvp = _kv(kv_len, B)
    rc = _load().fa_oracle_forward_m(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv,
                                     N, d, float(scale), int(bool(causal)), kvp, wl, wr, bmp,
                                     int(block), threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle forward failed ({rc})")
    return o, lse


def attention_fwd_rows(q, k, v, rows, scale, causal=False, kv_len=None, threads=None,
                       window=None):
    """Forward for selected query rows of one head; q, k, v are [N, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    wl, wr = _window(window)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    length = N if kv_len is None else int(kv_len)
    rc = _load().fa_oracle_forward_rows_v(_ptr(q), _ptr(k), _ptr(v), N, d, float(scale),
                                          int(bool(causal)), length, wl, wr,
                                          _ptr(rows, ctypes.c_int), int(rows.size), _ptr(o),
                                          _ptr(lse), threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle forward_rows failed ({rc})")
    return o, lse


def attention_bwd(q, k, v, do, scale, causal=False, kv_len=None, threads=None, window=None,
                  block_mask=None, block=128):
    """dQ [B,H,N,d], dK and dV [B,H_kv,N,d] (summed over each group's query
    heads) and D [B,H,N] (D_i = sum_j P_ij dP_ij); masks as in attention_fwd."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Hkv, N, d = _heads(q, k)
    assert v.shape == k.shape and do.shape == q.shape
    wl, wr = _window(window)
    bm, bmp = _block_mask(block_mask, N, block)
    dq = np.empty_like(q)
    dk, dv = np.empty_like(k), np.empty_like(k)
    D = np.empty((B, H, N), dtype=np.float64)
    kv, kvp = _kv(kv_len, B)
    rc = _load().fa_oracle_backward_m(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(D), B, H, Hkv, N, d, float(scale),
                                      int(bool(causal)), kvp, wl, wr, bmp, int(block),
                                      threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle backward failed ({rc})")
    return dq, dk, dv, D


def attention_decode(q, k, v, scale, causal=False, kv_len=None, threads=None, window=None):
    """O [B,H,Nq,d] and LSE [B,H,Nq] for Nq queries per head against Nk keys
    (k, v [B,H_kv,Nk,d]); query t of batch entry b sits at position
    kv_len[b] - Nq + t (kv_len None: Nk)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Nk, d) or v.shape != k.shape or Hkv < 1 or H % Hkv:
        raise ValueError(f"K/V shape {k.shape} does not match Q {q.shape}")
    wl, wr = _window(window)
    o = np.empty_like(q)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    kv, kvp = _kv(kv_len, B)
    rc = _load().fa_oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq,
                                  Nk, d, float(scale), int(bool(causal)), kvp, wl, wr,
                                  threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle decode failed ({rc})")
    return o, lse
