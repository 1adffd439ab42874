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


def _two_block_case(peak):
    """q = e_0; keys of block 0 score 0, keys of block 1 score `peak` (scale 1,
    unit Q/K scales); V random, quantised per head."""
    rng = np.random.default_rng(53)
    N, d = 256, 32
    q8 = np.zeros((1, 1, N, d), np.uint8)
    q8[..., 0] = 0x38                                   # q = e_0 (1.0)
    k8 = np.zeros((1, 1, N, d), np.uint8)
    k8[0, 0, 128:, 0] = F.e4m3_round(np.float32(peak))
    assert F.e4m3_decode(k8[0, 0, 135, 0]) == peak
    v = rng.standard_normal((1, N, d)).astype(np.float32)
    v8t, sv = F.quantize_v_transposed(v)
    return q8, k8, v8t.reshape(1, 1, d, -1), sv.reshape(1, 1)


@pytest.mark.parametrize("peak", [2.75, 3.0])
def test_slack_rule_closed_form(peak):
    """The recurrence worked by hand for the two-block case.  Block 0: m = 0,
    p = 1, P8 = E4M3(16) = 16.  Block 1 at peak 2.75 < 4 ln 2: m stays 0,
    p = e^2.75, P8 = E4M3(16 e^2.75).  At 3.0 > 4 ln 2: m moves to 3, block
    0's sums scale by e^-3, p = 1, P8 = 16.  O = sv (sum P8 V8) / (16 l)."""
    q8, k8, v8t, sv = _two_block_case(peak)
    ones = np.ones((1, 1, 2), np.float32)
    o, lse = F.attention_fp8(q8, ones, k8, ones, v8t, sv, 1.0, rows=[200])
    vc = F.e4m3_decode(v8t[0, 0]).T                     # [N, d] decoded codes
    s0, s1 = vc[:128].sum(0), vc[128:].sum(0)
    if peak < 4 * np.log(2):
        w1 = F.e4m3_decode(F.e4m3_round(np.float32(16 * np.exp(peak))))
        l = 128 + 128 * np.exp(peak)
        acc, m = 16 * s0 + w1 * s1, 0.0
    else:
        a = np.exp(-peak)
        l = 128 * a + 128
        acc, m = 16 * a * s0 + 16 * s1, peak
    np.testing.assert_allclose(o[0, 0, 200], float(sv[0, 0]) * acc / (16 * l), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 200], m + np.log(l), rtol=0, atol=1e-12)


@pytest.mark.parametrize("peak", [2.75, 3.0, 3.5])
def test_slack_keeps_16p_inside_e4m3(peak):
    """Block 0 scores 0; every key of block 1 scores `peak`: 2.75 < 4 ln 2
    (no rescale, so P reaches e^2.75 ~ 15.6 and 16 P ~ 250 must not
    saturate), 3.0 > 4 ln 2 (the reference moves).  Either way O must match
    exact attention of the dequantised inputs within E4M3's rounding of P."""
    N = 256
    q8, k8, v8t, sv = _two_block_case(peak)
    sq = np.ones((1, 1, 2), np.float32)
    sk = np.ones((1, 1, 2), np.float32)
    rows = [200, 255]                                   # see both blocks
    o, lse = F.attention_fp8(q8, sq, k8, sk, v8t, sv, 1.0, rows=rows)
    qd = F.e4m3_decode(q8)
    kd = F.e4m3_decode(k8)
    vd = F.e4m3_decode(v8t[..., :N]).transpose(0, 1, 3, 2) * sv[:, :, None, None]
    o_ref, lse_ref = oracle.attention_fwd(qd, kd, vd, 1.0)
    np.testing.assert_allclose(lse[0, 0, rows], lse_ref[0, 0, rows], rtol=0, atol=1e-10)
    # each P is normal here, so rounding it to E4M3 moves it by at most 2^-4
    # of itself: |dO| <= 2^-4 * sum_j softmax_j |v_j|, element by element
    s = (kd[0, 0] @ qd[0, 0, rows].T).T                  # exact scores of the rows
    w = np.exp(s - lse_ref[0, 0, rows][:, None])
    bound = 2.0 ** -4 * (w @ np.abs(vd[0, 0])) * (1 + 1e-9)
    assert np.all(np.abs(o[0, 0, rows] - o_ref[0, 0, rows]) <= bound)


# ---------------------------------------------------------------------------
# The parity bound of the E4M3 forward (tests/parity.py: fp8_o_bound).  The
# GPU kernel is compared with exact attention of the dequantised inputs under
# a bound that follows from E4M3's spacing alone.  Here, on the CPU, the
# step-by-step FP8 algorithm of oracle/fp8_ref.py is run with several
# choices of the rescale slack and the P multiplier that the pages leave
# open: every choice must stay within the bound (so the bound does not
# encode the kernel's tuning), the bound must not be vacuous, and planted
# mistakes must break it.
# ---------------------------------------------------------------------------
import parity as PB

TUNINGS = [(0.0, 256.0), (4 * np.log(2), 16.0), (8 * np.log(2), 1.0), (0.0, 1.0)]


def _fp8_case(gain, seed=61, B=1, H=2, N=300, d=32):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, H, N, d)) * gain).astype(np.float32)
    k = (rng.standard_normal((B, H, N, d)) * gain).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    q8, sq = F.quantize_rows(q.reshape(B * H, N, d))
    k8, sk = F.quantize_rows(k.reshape(B * H, N, d))
    v8t, sv = F.quantize_v_transposed(v.reshape(B * H, N, d))
    return {"q8": q8.reshape(B, H, N, d), "q_scale": sq.reshape(B, H, -1),
            "k8": k8.reshape(B, H, N, d), "k_scale": sk.reshape(B, H, -1),
            "v8t": v8t.reshape(B, H, d, -1), "v_scale": sv.reshape(B, H)}


def _ratio_to_bound(r, causal, slack, mult, v_scale_factor=1.0, block_mask=None):
    """max over elements of |O_fp8 - O_exact| / bound, for fp8_ref run with
    the given tuning (and planted changes), against exact attention of the
    dequantised inputs; also the share of visible keys whose weight sits
    below 2^-10 of its row's maximum (the subnormal regime at multiplier 16)."""
    N, d = r["q8"].shape[2], r["q8"].shape[3]
    scale = 1 / np.sqrt(d)
    qd, kd, vd = PB.dequantize(r, N)
    o, lse = F.attention_fp8(r["q8"], r["q_scale"], r["k8"], r["k_scale"], r["v8t"],
                             r["v_scale"] * v_scale_factor, scale, causal=causal, slack=slack,
                             p_mult=mult, block_mask=block_mask)
    worst, sub, vis = 0.0, 0, 0
    for h in range(r["q8"].shape[1]):
        Pw = PB.oracle_weights(qd[0, h], kd[0, h], scale, causal=causal)
        o_ref, lse_ref = oracle.attention_fwd(qd[:, h:h + 1], kd[:, h:h + 1], vd[:, h:h + 1],
                                              scale, causal=causal)
        bound = PB.fp8_o_bound(Pw, vd[0, h], o_ref[0, 0])
        worst = max(worst, float((np.abs(o[0, h] - o_ref[0, 0]) / bound).max()))
        rel = Pw / Pw.max(axis=1, keepdims=True)
        sub += int((rel[Pw > 0] < 2.0 ** -10).sum())
        vis += int((Pw > 0).sum())
        if block_mask is None:
            np.testing.assert_allclose(lse[0, h], lse_ref[0, 0], rtol=0, atol=1e-10)
    return worst, sub / vis


@pytest.mark.parametrize("gain", [1.0, 3.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("slack,mult", TUNINGS)
def test_fp8_bound_holds_for_any_tuning(gain, causal, slack, mult):
    """Slack 0 / 2^4 / 2^8 (in e-units 0, 4 ln 2, 8 ln 2) and multipliers
    256 / 16 / 1 all keep the largest P operand of a row in [1, 448] and the
    reference rising, so each must satisfy the E4M3 bound.  gain 1 puts
    nearly every weight in E4M3's normal range; gain 3 (scores of standard
    deviation about 9) puts most of them in the subnormal range, so both
    terms of the bound are exercised."""
    worst, sub = _ratio_to_bound(_fp8_case(gain), causal, slack, mult)
    assert worst <= 1.0, worst
    if gain == 3.0:
        assert sub > 0.5                 # mostly subnormal operands
    else:
        assert sub < 0.05                # mostly normal operands


def test_fp8_bound_is_not_vacuous():
    """The default tuning comes within a factor 2 of the bound somewhere in
    each regime, so the bound is not so loose that it pins nothing."""
    for gain in (1.0, 3.0):
        worst, _ = _ratio_to_bound(_fp8_case(gain), True, F.SLACK, F.P_MULT)
        assert worst >= 0.5, (gain, worst)


@pytest.mark.parametrize("gain", [1.0, 3.0])
def test_fp8_bound_catches_planted_mistakes(gain):
    """Planted in the oracle, on the CPU: a V scale off by a quarter, a
    dropped key block, and a multiplier (4096) that saturates E4M3.  Each
    must exceed the bound somewhere."""
    r = _fp8_case(gain)
    T = 3
    drop = np.ones((T, T), dtype=np.uint8)
    drop[2, 1] = 0
    assert _ratio_to_bound(r, True, F.SLACK, F.P_MULT, v_scale_factor=1.25)[0] > 1.0
    assert _ratio_to_bound(r, False, F.SLACK, F.P_MULT, block_mask=drop)[0] > 1.0
    assert _ratio_to_bound(r, True, 0.0, 4096.0)[0] > 1.0
