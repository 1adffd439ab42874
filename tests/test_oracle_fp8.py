"""Pins for the FP8 (E4M3) oracle in oracle/fp8_ref.py.

E4M3 rounding is checked against a brute-force nearest-code search with even
ties; the quantisers against their round-trip bound; the FP8 attention
against the exact (fp64, attn_oracle.c) attention of the dequantised inputs:
LSE must agree to fp64 precision (the row sum adds unrounded P) and O within
the E4M3 rounding of P, so a wrong scale, block order or mask fails."""
import numpy as np
import pytest

import oracle
from oracle import fp8_ref as F


def brute_round(x):
    vals = F.e4m3_values()
    finite = np.where(~np.isnan(vals))[0]
    out = []
    for v in np.asarray(x, dtype=np.float32).astype(np.float64):
        if v > 448:
            out.append(0x7E)
            continue
        if v < -448:
            out.append(0xFE)
            continue
        d = np.abs(vals[finite] - v)
        best = finite[d == d.min()]
        # ties: the code with an even mantissa; a zero carries the input's sign
        zero = 0x80 if np.signbit(v) else 0x00
        best = [c for c in best if vals[c] != 0 or c == zero] or list(best)
        even = [c for c in best if c % 2 == 0]
        out.append((even or best)[0])
    return np.array(out, dtype=np.uint8)


def test_known_codes():
    assert F.e4m3_decode(0x7E) == 448.0
    assert F.e4m3_decode(0x01) == 2.0 ** -9
    assert F.e4m3_decode(0x08) == 2.0 ** -6
    assert F.e4m3_decode(0x38) == 1.0
    assert F.e4m3_decode(0xB8) == -1.0
    assert np.isnan(F.e4m3_decode(0x7F))


def test_sign_is_kept_through_rounding_to_zero():
    assert F.e4m3_round(np.float32(-1e-6)) == 0x80
    assert F.e4m3_round(np.float32(1e-6)) == 0x00
    assert F.e4m3_round(np.float32(-0.0)) == 0x80


def test_rounding_matches_nearest_code_with_even_ties():
    rng = np.random.default_rng(50)
    vals = F.e4m3_values()
    finite = np.sort(np.unique(vals[~np.isnan(vals)]))
    mids = (finite[1:] + finite[:-1]) / 2                  # every tie
    x = np.concatenate([rng.standard_normal(3000) * 10, rng.standard_normal(1000) * 0.01,
                        mids, -mids, [500.0, -1000.0, 447.0, 460.0, 0.0, -0.0, 2.0 ** -11,
                                      -2.0 ** -10, -2.0 ** -11, -1e-7]])
    x = x.astype(np.float32)
    got = F.e4m3_round(x)
    ref = brute_round(x)
    assert np.array_equal(got, ref), (x[got != ref][:10], got[got != ref][:10], ref[got != ref][:10])


def test_quantize_round_trip_bound():
    rng = np.random.default_rng(51)
    x = (rng.standard_normal((2, 300, 64)) * 3).astype(np.float32)
    codes, sc = F.quantize_rows(x)
    deq = F.e4m3_decode(codes) * np.repeat(sc, 128, axis=1)[:, :300, None]
    # within half a quantum of the block's E4M3 grid: relative 2^-4 above the
    # smallest normal, absolute 2^-10 * scale below it
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * np.repeat(sc, 128, axis=1)[:, :300, None])
    assert np.all(err <= bound * (1 + 1e-6))
    v8t, sv = F.quantize_v_transposed(x)
    assert v8t.shape == (2, 64, 384) and np.all(v8t[:, :, 300:] == 0)
    deqv = F.e4m3_decode(v8t[:, :, :300]).transpose(0, 2, 1) * sv[:, None, None]
    assert np.all(np.abs(deqv - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sv[:, None, None]) * (1 + 1e-6))


@pytest.mark.parametrize("causal,kv,Hkv,window", [(False, None, 2, None), (True, None, 2, None),
                                                  (True, [150, 300], 1, None),
                                                  (True, None, 1, (70, 0)),
                                                  (False, [200, 300], 2, (40, 130))])
def test_fp8_attention_against_exact_attention_of_dequantised_inputs(causal, kv, Hkv, window):
    rng = np.random.default_rng(52)
    B, H, N, d = 2, 2, 300, 32
    q = (rng.standard_normal((B, H, N, d)) * 2).astype(np.float32)
    k = (rng.standard_normal((B, Hkv, N, d)) * 2).astype(np.float32)
    v = rng.standard_normal((B, Hkv, N, d)).astype(np.float32)
    q8, sq = F.quantize_rows(q.reshape(B * H, N, d))
    k8, sk = F.quantize_rows(k.reshape(B * Hkv, N, d))
    v8t, sv = F.quantize_v_transposed(v.reshape(B * Hkv, N, d))
    q8, sq = q8.reshape(B, H, N, d), sq.reshape(B, H, -1)
    k8, sk = k8.reshape(B, Hkv, N, d), sk.reshape(B, Hkv, -1)
    v8t, sv = v8t.reshape(B, Hkv, d, -1), sv.reshape(B, Hkv)
    scale = 1 / np.sqrt(d)
    o, lse = F.attention_fp8(q8, sq, k8, sk, v8t, sv, scale, causal=causal, kv_len=kv,
                             window=window)
    qd = F.e4m3_decode(q8) * np.repeat(sq, 128, axis=2)[:, :, :N, None]
    kd = F.e4m3_decode(k8) * np.repeat(sk, 128, axis=2)[:, :, :N, None]
    vd = F.e4m3_decode(v8t[..., :N]).transpose(0, 1, 3, 2) * sv[:, :, None, None]
    o_ref, lse_ref = oracle.attention_fwd(qd, kd, vd, scale, causal=causal, kv_len=kv,
                                          window=window)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-10)
    err = np.abs(o - o_ref)
    assert err.max() <= 2.0 ** -4 * np.abs(vd).max()           # P rounded to E4M3
    assert err.mean() <= 2e-3 * np.abs(vd).max()
