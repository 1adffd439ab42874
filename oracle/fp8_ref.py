"""FP8 (E4M3) attention forward, as the pages describe it, in numpy.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only the tests, the
smoke check and the benchmark's CPU legs use it.

"4. FlashAttention 深度剖析" 4.5.4 gives the method in three points: E4M3
for the forward, a scale per K block applied when the block is loaded, and
FP32 accumulation of the FP8 products.  It does not fix the rest; the
readings below are also the GPU kernel's.  The GPU path is not
checked against this file: its parity test compares it with exact attention
(attn_oracle.c) of the dequantised inputs under a bound derived from E4M3's
spacing, which any slack and multiplier in range satisfy.  This file serves
the CPU pins of that bound (it shows the bound holds for several tunings and
fails for planted mistakes) and is a step-by-step diagnostic:

* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits, subnormals, largest
  finite 448, no infinities.  Conversion from fp32 rounds to nearest, ties
  to even, saturates to +-448, and keeps the sign (a negative value that
  rounds to zero becomes -0, as IEEE conversions do).
* Q is scaled per 128-row tile of a head, K per 128-key block of a K/V head,
  V per K/V head: scale = amax / 448 (fp32), stored value = E4M3(x * (448 /
  amax)) with that product and quotient rounded to fp32; an all-zero block
  has scale 1.  V gets one scale per head so that the P V sum can be scaled
  once at the end.
* The softmax is the block-online recurrence of 4.3.2 over 128-key blocks
  in order.  Within a block, S = sq * sk * (Q8 K8^T) * scale.  The reference
  maximum m starts at the first block's maximum and is raised to a block's
  maximum only when that exceeds m by more than 4 ln 2 (a factor 2^4), so
  P = exp(S - m) <= 16 and is stored as E4M3(16 * P) <= 256 for the P V
  product; the row sum l adds the unrounded P.  O = sv * (sum of P8 V8) /
  (16 * l), LSE = m + ln l.  (16 P keeps the normal range, relative to the
  row maximum, that 256 P has when m follows every new maximum; the slack
  spares the rescale of O on most blocks.)

Unlike attn_oracle.c this is an algorithm, not a definition: its blocks and
rounding are part of the result, so they are written out step by step.
"""
import numpy as np

E4M3_MAX = 448.0
BLOCK = 128
SLACK = 4.0 * np.log(2.0)     # the reference maximum moves past 2^4 growth
P_MULT = 16.0                 # E4M3 operand = 16 P


def e4m3_values():
    """The value of every E4M3 code (NaN codes 0x7f and 0xff as nan)."""
    codes = np.arange(256, dtype=np.int64)
    s = np.where(codes >> 7, -1.0, 1.0)
    e = (codes >> 3) & 15
    m = codes & 7
    v = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    v = s * v
    v[(codes & 0x7F) == 0x7F] = np.nan
    return v


_VALUES = e4m3_values()


def e4m3_round(x):
    """uint8 E4M3 codes of fp32 values x: round to nearest, ties to even,
    saturating to +-448.  Written from the format's definition: the spacing
    of representable magnitudes is 2^(max(e, -6) - 3) for |x| in [2^e, 2^(e+1))."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    q = np.round(a / quantum) * quantum          # numpy rounds half to even
    q = np.minimum(q, E4M3_MAX)
    q = np.where(a > 0, q, 0.0)
    # encode the (now representable) magnitude
    codes = np.zeros(q.shape, dtype=np.int64)
    normal = q >= 2.0 ** -6
    en = np.floor(np.log2(np.where(normal, q, 1.0)))
    mant = np.where(normal, q / np.ldexp(1.0, en.astype(np.int64)) - 1.0, q / 2.0 ** -6)
    mcode = np.round(mant * 8).astype(np.int64)
    ecode = np.where(normal, en.astype(np.int64) + 7, 0)
    codes = (ecode << 3) | mcode
    codes = np.where(np.signbit(x), codes | 0x80, codes)
    return codes.astype(np.uint8)


def e4m3_decode(codes):
    return _VALUES[np.asarray(codes, dtype=np.int64)]


def block_scale(amax):
    """(dequantisation scale, multiplier) in fp32 for a block with amax."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0), np.float32(1.0)
    return np.float32(amax / np.float32(E4M3_MAX)), np.float32(np.float32(E4M3_MAX) / amax)


def quantize_rows(x):
    """x [G, N, d] (fp32-representable) -> (codes [G, N, d] uint8, scales
    [G, ceil(N/128)] fp32), one scale per 128-row block of each of the G
    heads."""
    x = np.asarray(x, dtype=np.float32)
    G, N, d = x.shape
    nb = -(-N // BLOCK)
    codes = np.zeros((G, N, d), dtype=np.uint8)
    scales = np.zeros((G, nb), dtype=np.float32)
    for g in range(G):
        for b in range(nb):
            blk = x[g, b * BLOCK:(b + 1) * BLOCK]
            s, mul = block_scale(np.abs(blk).max())
            scales[g, b] = s
            codes[g, b * BLOCK:(b + 1) * BLOCK] = e4m3_round(blk * mul)
    return codes, scales


def quantize_v_transposed(v):
    """v [G, N, d] -> (codes [G, d, Npad] uint8 with keys contiguous and
    zero padding up to a multiple of 128, scales [G] fp32), one scale per head."""
    v = np.asarray(v, dtype=np.float32)
    G, N, d = v.shape
    npad = -(-N // BLOCK) * BLOCK
    codes = np.zeros((G, d, npad), dtype=np.uint8)
    scales = np.zeros(G, dtype=np.float32)
    for g in range(G):
        s, mul = block_scale(np.abs(v[g]).max())
        scales[g] = s
        codes[g, :, :N] = e4m3_round(v[g] * mul).T
    return codes, scales


def attention_fp8(q8, sq, k8, sk, v8t, sv, scale, causal=False, kv_len=None, H_kv=None,
                  rows=None, window=None, block_mask=None, slack=SLACK, p_mult=P_MULT):
    """O [B,H,N,d] and LSE [B,H,N] of the FP8 forward, step by step.

    q8 [B,H,N,d] codes with sq [B,H,ceil(N/128)]; k8 [B,H_kv,N,d] with
    sk [B,H_kv,ceil(N/128)]; v8t [B,H_kv,d,Npad] with sv [B,H_kv].  rows: a
    list of query rows to compute (the others are left 0 / -inf).  window:
    (left, right), query i sees keys i-left..i+right (-1: unbounded side),
    the same visibility rule as the bf16 oracle; causal caps right at 0.
    block_mask: [nb, nb] (or None), zero where key block j is skipped for
    the rows of query block i // 128 (Block-Sparse FlashAttention, "炉案与百步
    之外的仓库…" 第八部分): the recurrence passes over that block.
    slack, p_mult: the rescale slack (natural-log units) and the power-of-two
    multiplier of the E4M3 P operand.  The pages fix neither; the defaults
    are the readings above, and the tests also run other choices (0 and 256,
    8 ln 2 and 1) to show that their parity bound does not depend on them."""
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if causal:
        wr = 0
    B, H, N, d = q8.shape
    Hkv = k8.shape[1] if H_kv is None else H_kv
    G = H // Hkv
    Q = e4m3_decode(q8)
    K = e4m3_decode(k8)
    V = e4m3_decode(v8t)
    nb = -(-N // BLOCK)
    O = np.zeros((B, H, N, d))
    LSE = np.full((B, H, N), -np.inf)
    for b in range(B):
        ln = N if kv_len is None else int(min(max(kv_len[b], 0), N))
        for h in range(H):
            hk = h // G
            for i in (range(N) if rows is None else rows):
                m = -np.inf
                l = 0.0
                acc = np.zeros(d)
                sqi = float(sq[b, h, i // BLOCK])
                for j in range(nb):
                    if block_mask is not None and not block_mask[i // BLOCK][j]:
                        continue
                    k0, k1 = j * BLOCK, min((j + 1) * BLOCK, N)
                    lo = k0 if wl < 0 else max(k0, i - wl)
                    hi = min(k1, ln, k1 if wr < 0 else i + wr + 1)
                    if hi <= lo:
                        continue
                    s = (K[b, hk, lo:hi] @ Q[b, h, i]) * (sqi * float(sk[b, hk, j])) * scale
                    mb = s.max()
                    if m == -np.inf:
                        m = mb
                    elif mb > m + slack:               # raise the reference to the new max
                        alpha = np.exp(m - mb)
                        acc *= alpha
                        l *= alpha
                        m = mb
                    p = np.exp(s - m)
                    p8 = e4m3_decode(e4m3_round((p * p_mult).astype(np.float32)))
                    l += p.sum()
                    acc += V[b, hk, :, lo:hi] @ p8
                if l > 0:
                    O[b, h, i] = float(sv[b, hk]) * acc / (p_mult * l)
                    LSE[b, h, i] = m + np.log(l)
    return O, LSE
