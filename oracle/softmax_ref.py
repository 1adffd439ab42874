"""The pages' softmax recurrences in numpy float64.

TEST INFRASTRUCTURE (part of the oracle; see ``oracle/__init__.py``).

Each function follows one passage, in the notation of that passage:

* ``safe_softmax_3pass``   - "4. FlashAttention 深度剖析" (llm-training-tutorial),
  section 4.2.1: m = max_j x_j, d = sum_j e^(x_j - m), y_j = e^(x_j - m) / d.
* ``online_normalizer``     - same page, section 4.2.2: the two-pass version whose
  first pass carries (m, d) together and rescales d by e^(m_old - m_new).
* ``online_softmax_times_v`` - section 4.2.3: one pass that carries the
  unnormalised output O~ and l, divided once at the end.
* ``block_state`` / ``merge`` - section 4.2.4: the per-block triple
  (m, l, O~) and the associative merge of two triples.
* ``online_block_update``   - "注意力为什么受限于显存带宽…" (magicnetworld), section
  六: the row-block update of (m, l, O) when block j of scores arrives.
* ``tiled_forward``         - llm-training-tutorial section 4.3.2: outer loop over
  Q row blocks, inner loop over K/V column blocks, online update, divide by l
  at the end and save L = m + log l; causal blocks entirely above the
  diagonal are skipped.

Masked scores are -inf.  Where a row has seen only -inf so far its running
maximum is -inf; the rescale factor is then taken as 1 (there is nothing to
rescale) instead of the undefined e^(-inf - -inf).
"""
import numpy as np


def safe_softmax_3pass(x):
    """Three passes over x: max, sum of exp(x - max), divide.  Returns (y, m, d)."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)                       # pass 1
    e = np.exp(x - m)
    d = np.sum(e)                       # pass 2
    return e / d, m, d                  # pass 3


def online_normalizer(x, trajectory=False):
    """Carry (m, d) through one scan of x (section 4.2.2).

    Returns the final (m, d); with ``trajectory`` also the list of (m, d)
    after each element.
    """
    m, d = -np.inf, 0.0
    traj = []
    for xi in np.asarray(x, dtype=np.float64):
        m_new = max(m, xi)
        scale_old = np.exp(m - m_new) if m != -np.inf else 0.0
        d = d * scale_old + np.exp(xi - m_new)
        m = m_new
        traj.append((m, d))
    return (m, d, traj) if trajectory else (m, d)


def online_softmax_times_v(x, V):
    """One pass over (x_i, v_i) keeping O~ and l; O = O~ / l (section 4.2.3).

    Returns (O, m, l).
    """
    V = np.asarray(V, dtype=np.float64)
    m, l = -np.inf, 0.0
    O_t = np.zeros(V.shape[1], dtype=np.float64)
    for xi, vi in zip(np.asarray(x, dtype=np.float64), V):
        m_new = max(m, xi)
        c = np.exp(m - m_new) if m != -np.inf else 0.0
        p = np.exp(xi - m_new)
        O_t = O_t * c + p * vi
        l = l * c + p
        m = m_new
    return O_t / l, m, l


def block_state(x, V):
    """(m, l, O~) of one block of scores x with its value rows V (section 4.2.4)."""
    x = np.asarray(x, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m = np.max(x)
    e = np.exp(x - m)
    return m, np.sum(e), e @ V


def merge(a, b):
    """Merge two block states (m, l, O~) (section 4.2.4); associative."""
    m_a, l_a, O_a = a
    m_b, l_b, O_b = b
    m = max(m_a, m_b)
    e_a = np.exp(m_a - m) if m_a != -np.inf else 0.0
    e_b = np.exp(m_b - m) if m_b != -np.inf else 0.0
    return m, l_a * e_a + l_b * e_b, O_a * e_a + O_b * e_b


def online_block_update(m, l, O, S_j, V_j):
    """One step of the row-block recurrence of magicnetworld section 六.

    m, l: [rows]; O: [rows, d] (unnormalised); S_j: [rows, cols] scores of
    block j (-inf where masked); V_j: [cols, d].  Returns the new (m, l, O).
    """
    m_blk = np.max(S_j, axis=1)
    m_new = np.maximum(m, m_blk)
    seen = m_new != -np.inf
    alpha = np.where(seen, np.exp(np.where(seen, m - m_new, 0.0)), 1.0)
    P = np.where(seen[:, None], np.exp(S_j - np.where(seen, m_new, 0.0)[:, None]), 0.0)
    l_new = alpha * l + P.sum(axis=1)
    O_new = alpha[:, None] * O + P @ V_j
    return m_new, l_new, O_new


def tiled_forward(q, k, v, scale, causal=False, kv_len=None, Br=16, Bc=16):
    """Tiled forward of one head (section 4.3.2).  q, k, v: [N, d].

    Returns (O [N, d], L [N]) with L = m + log(l) in natural-log units of
    scale * q.k.  ``kv_len``: keys j >= kv_len are masked for every query.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    N, d = q.shape
    length = N if kv_len is None else int(kv_len)
    O = np.zeros((N, d))
    L = np.zeros(N)
    for i0 in range(0, N, Br):
        rows = np.arange(i0, min(i0 + Br, N))
        m = np.full(rows.size, -np.inf)
        l = np.zeros(rows.size)
        O_i = np.zeros((rows.size, d))
        for j0 in range(0, N, Bc):
            if causal and j0 > rows[-1]:
                break                                   # block entirely above the diagonal
            cols = np.arange(j0, min(j0 + Bc, N))
            S = scale * (q[rows] @ k[cols].T)
            mask = cols[None, :] >= length
            if causal:
                mask = mask | (cols[None, :] > rows[:, None])
            S = np.where(mask, -np.inf, S)
            m, l, O_i = online_block_update(m, l, O_i, S, v[cols])
        O[rows] = O_i / l[:, None]
        L[rows] = m + np.log(l)
    return O, L
