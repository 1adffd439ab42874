"""Pins for the softmax recurrences of the oracle (oracle/softmax_ref.py).

Checked against the numbers the pages print for two worked examples
(tests/golden/softmax_worked_examples.json), against the three-pass safe
softmax that the recurrences must equal (the induction argument of
llm-training-tutorial section 4.2.2), and against each other.
"""
import json
import os

import numpy as np
import pytest

from oracle import softmax_ref as sr
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_worked_examples.json")


def _example(ex_id):
    with open(GOLDEN) as f:
        for ex in json.load(f)["examples"]:
            if ex["id"] == ex_id:
                return ex
    raise KeyError(ex_id)


def test_worked_example_7_4_3_three_pass():
    ex = _example("scores_7_4_3_then_9")
    y, m, d = sr.safe_softmax_3pass(ex["scores_first"])
    tol = ex["tol"]
    assert m == 7
    assert abs(d - ex["denominator_first"]) <= tol
    np.testing.assert_allclose(np.exp(np.array(ex["scores_first"]) - m),
                               ex["exp_shifted_first"], atol=tol)
    np.testing.assert_allclose(y, ex["weights_first"], atol=tol)


def test_worked_example_7_4_3_then_9_online():
    ex = _example("scores_7_4_3_then_9")
    xs = ex["scores_first"] + [ex["score_added"]]
    m, d, traj = sr.online_normalizer(xs, trajectory=True)
    tol = ex["tol"]
    assert traj[2][0] == 7 and abs(traj[2][1] - ex["denominator_first"]) <= tol
    assert m == 9 and abs(d - ex["denominator_after"]) <= tol
    # the page's identity: new denominator = old * exp(old max - new max) + exp(new - new max)
    s1 = traj[2][1]
    assert abs(s1 * np.exp(7 - 9) + np.exp(9 - 9) - d) <= 1e-15
    # and the same denominator recomputed from scratch with the new maximum
    np.testing.assert_allclose(np.exp(np.array(xs) - 9), ex["exp_shifted_after"], atol=tol)
    assert abs(sr.safe_softmax_3pass(xs)[2] - d) <= 1e-14


def test_worked_example_two_blocks_merge_and_row_update():
    ex = _example("two_blocks_3_1_then_5_2")
    a = sr.block_state(ex["block_1"], np.zeros((2, 1)))
    b = sr.block_state(ex["block_2"], np.zeros((2, 1)))
    assert a[0] == ex["m_after_block_1"]
    assert abs(a[1] - ex["l_after_block_1"]) <= ex["tol_3dp"]
    assert abs(a[1] * np.exp(a[0] - 5) - ex["l_block_1_rescaled"]) <= ex["tol_4dp"]
    assert abs(b[1] - ex["block_2_exp_sum"]) <= ex["tol_4dp"]
    m, l, _ = sr.merge(a, b)
    assert m == ex["m_after_block_2"] and abs(l - ex["l_after_block_2"]) <= ex["tol_4dp"]
    # the same two steps through the row-block recurrence of section 六
    mr, lr, Or = np.array([-np.inf]), np.zeros(1), np.zeros((1, 1))
    mr, lr, Or = sr.online_block_update(mr, lr, Or, np.array([ex["block_1"]], float), np.ones((2, 1)))
    assert abs(lr[0] - ex["l_after_block_1"]) <= ex["tol_3dp"]
    mr, lr, Or = sr.online_block_update(mr, lr, Or, np.array([ex["block_2"]], float), np.ones((2, 1)))
    assert mr[0] == 5 and abs(lr[0] - ex["l_after_block_2"]) <= ex["tol_4dp"]
    assert abs(Or[0, 0] - lr[0]) <= 1e-15       # V = 1: O~ equals l


def _vectors(rng):
    yield rng.standard_normal(1)
    yield rng.standard_normal(37) * 5
    yield np.arange(50, dtype=float)             # max moves at every element
    yield -np.arange(50, dtype=float)            # max never moves after the first
    yield rng.uniform(-1000, 1000, 200)          # would overflow exp without the max
    yield np.full(17, 3.25)                      # ties


def test_online_normalizer_equals_three_pass():
    rng = np.random.default_rng(0)
    for x in _vectors(rng):
        m, d = sr.online_normalizer(x)
        _, m3, d3 = sr.safe_softmax_3pass(x)
        assert m == m3
        assert abs(d - d3) <= 1e-12 * d3


def test_one_pass_softmax_times_v_equals_three_pass():
    rng = np.random.default_rng(1)
    for x in _vectors(rng):
        V = rng.standard_normal((x.size, 6))
        O, m, l = sr.online_softmax_times_v(x, V)
        y, m3, d3 = sr.safe_softmax_3pass(x)
        np.testing.assert_allclose(O, y @ V, rtol=0, atol=1e-12 * np.abs(V).max())
        assert m == m3 and abs(l - d3) <= 1e-12 * d3


def _random_tree_merge(states, rng):
    states = list(states)
    while len(states) > 1:
        i = int(rng.integers(0, len(states) - 1))
        states[i:i + 2] = [sr.merge(states[i], states[i + 1])]
    return states[0]


def test_block_merge_is_associative_over_random_splits_and_trees():
    rng = np.random.default_rng(2)
    for trial in range(40):
        n = int(rng.integers(2, 90))
        x = rng.standard_normal(n) * rng.choice([1.0, 10.0, 300.0])
        V = rng.standard_normal((n, 5))
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(n - 1, int(rng.integers(1, 8))),
                                  replace=False))
        blocks = np.split(np.arange(n), cuts)
        states = [sr.block_state(x[b], V[b]) for b in blocks]
        whole = sr.block_state(x, V)
        for _ in range(3):
            m, l, O = _random_tree_merge(states, rng)
            assert m == whole[0]
            assert abs(l - whole[1]) <= 1e-12 * whole[1]
            np.testing.assert_allclose(O, whole[2], rtol=1e-12, atol=1e-12 * np.abs(whole[2]).max())
        y, _, _ = sr.safe_softmax_3pass(x)
        np.testing.assert_allclose(O / l, y @ V, rtol=0, atol=1e-12 * np.abs(V).max())


def test_merge_identity_element():
    rng = np.random.default_rng(3)
    s = sr.block_state(rng.standard_normal(9), rng.standard_normal((9, 3)))
    empty = (-np.inf, 0.0, np.zeros(3))
    for got in (sr.merge(s, empty), sr.merge(empty, s)):
        assert got[0] == s[0] and got[1] == s[1]
        np.testing.assert_array_equal(got[2], s[2])


@pytest.mark.parametrize("N,d,causal,kv,Br,Bc", [
    (33, 8, False, None, 8, 8),
    (33, 8, True, None, 8, 16),
    (50, 4, False, 27, 16, 8),
    (50, 4, True, 31, 7, 5),
    (1, 3, True, None, 4, 4),
])
def test_tiled_forward_equals_definition(N, d, causal, kv, Br, Bc):
    rng = np.random.default_rng(N * 7 + d)
    q, k, v = (rng.standard_normal((N, d)) * 2 for _ in range(3))
    scale = 0.7
    O, L = sr.tiled_forward(q, k, v, scale, causal=causal, kv_len=kv, Br=Br, Bc=Bc)
    Oref, Lref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale,
                                      causal=causal, kv_len=None if kv is None else [kv])
    np.testing.assert_allclose(O, Oref[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lref[0, 0], rtol=0, atol=1e-12)
