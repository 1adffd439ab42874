"""Host-side checks of the causal schedule planner (no GPU needed).

A causal work item costs in proportion to its distance from one end of the
sequence: query tile m of the forward sees m + 1 key blocks, key block n of
the backward is seen by 2 (T - n) query steps.  The kernels pair items into
equal units that go round-robin over the CTAs (unit u on CTA u % G), except
for the last `heads` heads, whose single items the host places, longest
first, on the least-loaded CTA.  The kernels walk each CTA's round-robin
units, then its row of the table.

These tests call the planner in the built library and check the plan it
returns:
- the paired units and the table together hold every (head, half, block)
  exactly once;
- rows are -1-terminated and within their capacity;
- each CTA's items run longest first;
- the plan beats plain round-robin of pairs.

The block-sparse planner (plan_mask_tail) gets the same checks with single
items dealt round-robin, plus its costs: the computed blocks of each item,
counted position by position in the mask and the window.
"""
import ctypes

import pytest

from exact_attention_04_gb300 import build as fabuild
from exact_attention_04_gb300 import fa

TAIL_CTAS, TAIL_ITEMS = 160, 8
PLAN = "_ZN2fa16plan_causal_tailEiiiibxPNS_9TailTableE"  # fa::plan_causal_tail, Itanium ABI


class TailTable(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("item", (ctypes.c_int * TAIL_ITEMS) * TAIL_CTAS)]


@pytest.fixture(scope="module")
def plan():
    fabuild.build()
    lib = fa.load()
    f = getattr(lib, PLAN)
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_bool,
                  ctypes.c_longlong, ctypes.POINTER(TailTable)]
    f.restype = None

    def run(BH, T, nsplit, G, fwd, head_bytes=0):
        t = TailTable()
        f(BH, T, nsplit, G, fwd, head_bytes, ctypes.byref(t))
        return t
    return run


def cost(T, fwd, blk):
    return (blk + 1 if fwd else 2 * (T - blk)) + (3 if fwd else 4)


def items_of_pair(T, pp):
    return [pp] if pp == T - 1 - pp else [pp, T - 1 - pp]


def walk(t, BH, T, nsplit, G, fwd):
    """Each CTA's items as the kernels walk them: (head, half, block) lists."""
    P = (T + 1) // 2
    units = (BH - t.heads) * P * nsplit
    per_cta = [[] for _ in range(G)]
    for u in range(units):
        bh, rem = divmod(u, P * nsplit)
        pp, h = divmod(rem, nsplit)
        for n in items_of_pair(T, pp):
            per_cta[u % G].append((bh, h, n))
    for c in range(G):
        row = list(t.item[c]) if c < TAIL_CTAS else []
        seen_end = False
        for e in row:
            if e < 0:
                seen_end = True
                continue
            assert not seen_end, f"CTA {c}: an entry after the end of its row"
            per_cta[c].append((e >> 12, (e >> 11) & 1, e & 2047))
    return per_cta


SHAPES = [
    # BH, T, nsplit, G, fwd
    (32, 64, 1, 152, True),      # B=2, H=16, N=8192 forward
    (32, 64, 1, 152, False),     # its backward, d = 128
    (32, 64, 2, 152, False),     # d = 256: two halves of the head dimension
    (64, 64, 1, 152, True),      # B=2, H=32
    (16, 64, 1, 152, False),     # GQA: B=2, H_kv=8
    (96, 8, 1, 152, True),       # B=8, H=12, N=1024
    (1, 2, 1, 2, True),          # B=1, H=1, N=256: two tiles, two CTAs
    (4, 5, 1, 20, False),        # odd T: the middle pair is a single item
    (2, 3, 2, 12, False),
    (8, 256, 1, 152, True),      # long sequence, few heads
]


@pytest.mark.parametrize("BH,T,nsplit,G,fwd", SHAPES)
def test_plan_covers_every_item_once(plan, BH, T, nsplit, G, fwd):
    t = plan(BH, T, nsplit, G, fwd)
    assert 0 <= t.heads <= BH
    got = sorted(x for c in walk(t, BH, T, nsplit, G, fwd) for x in c)
    want = sorted((bh, h, n) for bh in range(BH) for h in range(nsplit) for n in range(T))
    assert got == want
    for c in range(TAIL_CTAS):
        for e in t.item[c]:
            if e >= 0:
                assert e >> 12 >= BH - t.heads, "a tail item outside the tail heads"


@pytest.mark.parametrize("BH,T,nsplit,G,fwd", SHAPES)
def test_tail_items_run_longest_first(plan, BH, T, nsplit, G, fwd):
    t = plan(BH, T, nsplit, G, fwd)
    for c in range(min(G, TAIL_CTAS)):
        costs = [cost(T, fwd, e & 2047) for e in t.item[c] if e >= 0]
        assert costs == sorted(costs, reverse=True)


@pytest.mark.parametrize("BH,T,nsplit,G,fwd,bound", [
    (32, 64, 1, 152, True, 0.015), (32, 64, 1, 152, False, 0.015),
    (64, 64, 1, 152, True, 0.015), (96, 8, 1, 152, True, 0.1)])
def test_plan_balances_the_causal_step(plan, BH, T, nsplit, G, fwd, bound):
    """The busiest CTA's work within `bound` of the mean, where plain
    round-robin of equal pairs leaves the last round part-empty (about 4 %
    above the mean at B=2, H=16, N=8192 and 19 % at B=8, H=12, N=1024, where
    an item costs 4 to 11 against a mean of 38 a CTA)."""
    t = plan(BH, T, nsplit, G, fwd)
    assert t.heads > 0
    loads = [sum(cost(T, fwd, n) for _, _, n in c) for c in walk(t, BH, T, nsplit, G, fwd)]
    mean = sum(loads) / G
    assert max(loads) <= mean * (1 + bound)
    P = (T + 1) // 2
    rr = [0] * G
    for u in range(BH * P * nsplit):
        rr[u % G] += sum(cost(T, fwd, n) for n in items_of_pair(T, (u // nsplit) % P))
    assert max(loads) < max(rr)


def test_tail_heads_fit_their_l2_share(plan):
    """The tail runs its heads at once: at most 64 MB of what they share."""
    mb = 1 << 20
    assert plan(32, 64, 1, 152, True, 4 * mb).heads == 14      # K+V of N=8192, d=128: 56 MB
    assert plan(32, 64, 1, 152, True, 8 * mb).heads == 8       # d = 256
    assert plan(32, 64, 1, 152, True, 100 * mb).heads == 1
    assert plan(32, 64, 1, 152, True, 0).heads == 14           # no limit: six items a CTA


def test_plan_declines_what_the_table_cannot_hold(plan):
    assert plan(32, 64, 1, TAIL_CTAS + 1, True).heads == 0     # too many CTAs
    assert plan(1, 4096, 1, 152, True).heads == 0              # blocks past 2047
    t = plan(32, 64, 1, 152, True)
    assert all(t.item[c][k] == -1 for c in range(152, TAIL_CTAS) for k in range(TAIL_ITEMS))


def test_plan_is_repeatable_across_interleaved_calls(plan):
    """Plans are memoised per argument set; interleaved calls with other
    arguments must not hand back another shape's table."""
    shapes = [(32, 64, 1, 152, True, 4 << 20), (32, 64, 1, 152, False, 4 << 20),
              (96, 8, 1, 152, True, 1 << 20), (32, 64, 2, 152, False, 8 << 20),
              (16, 64, 1, 152, False, 16 << 20)]
    first = [plan(*s) for s in shapes]
    for _ in range(3):                      # more calls than the memo holds between repeats
        for s, t0 in zip(shapes[::-1], first[::-1]):
            t = plan(*s)
            assert t.heads == t0.heads
            assert all(list(t.item[c]) == list(t0.item[c]) for c in range(TAIL_CTAS))


# ---- block-sparse schedules: single items, costed by the mask ----

MASK_PLAN = "_ZN2fa14plan_mask_tailEPKhiiiibiiixPNS_9TailTableE"   # fa::plan_mask_tail
UNB = -1                                  # an unbounded window side, as the binding passes it


@pytest.fixture(scope="module")
def mask_plan():
    fabuild.build()
    lib = fa.load()
    f = getattr(lib, MASK_PLAN)
    f.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_bool, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong,
                  ctypes.POINTER(TailTable)]
    f.restype = None

    def run(bm, BH, nsplit, G, fwd, N, wl=1 << 30, wr=1 << 30, head_bytes=0):
        t = TailTable()
        f(None if bm is None else bytes(bm.astype("uint8").ravel()), BH, bm.shape[0] if bm is not None else 1,
          nsplit, G, fwd, N, wl, wr, head_bytes, ctypes.byref(t))
        return t
    return run


def mask_costs(bm, fwd, N, wl, wr):
    """Item costs counted position by position: a block is computed for an
    item when its mask entry is set and some (query, key) pair of the two
    blocks is inside the window."""
    T = bm.shape[0]
    out = []
    for b in range(T):
        n = 0
        for o in range(T):
            a, c = (b, o) if fwd else (o, b)          # (query block, key block)
            seen = any(i - wl <= j <= i + wr
                       for i in range(128 * a, min(128 * a + 128, N))
                       for j in range(128 * c, min(128 * c + 128, N)))
            n += bool(bm[a, c]) and seen
        out.append((n if fwd else 2 * n) + (3 if fwd else 4))
    return out


def walk_single(t, BH, T, nsplit, G):
    """Each CTA's items as the kernels walk them without pairing: unit u is
    (head u // (T nsplit), block (u // nsplit) % T, half u % nsplit) on CTA
    u % G, then the CTA's tail row."""
    per_cta = [[] for _ in range(G)]
    for u in range((BH - t.heads) * T * nsplit):
        bh, rem = divmod(u, T * nsplit)
        n, h = divmod(rem, nsplit)
        per_cta[u % G].append((bh, h, n))
    for c in range(min(G, TAIL_CTAS)):
        row = list(t.item[c])
        live = [e for e in row if e >= 0]
        assert row[:len(live)] == live, f"CTA {c}: an entry after the end of its row"
        per_cta[c] += [(e >> 12, (e >> 11) & 1, e & 2047) for e in live]
    return per_cta


def bench_mask(T=64, seed=12):
    from exact_attention_04_gb300.workloads import block_sparse_mask
    return block_sparse_mask(T, seed=seed)


MASK_SHAPES = [
    # BH, nsplit, G, fwd
    (32, 1, 152, True),       # B=2, H=16, N=8192 forward
    (32, 1, 152, False),      # its backward
    (32, 2, 152, False),      # d = 256
    (16, 1, 152, False),      # GQA K/V heads
    (3, 1, 20, True),
]


@pytest.mark.parametrize("BH,nsplit,G,fwd", MASK_SHAPES)
def test_mask_plan_covers_every_item_once(mask_plan, BH, nsplit, G, fwd):
    bm = bench_mask()
    T = bm.shape[0]
    t = mask_plan(bm, BH, nsplit, G, fwd, 128 * T)
    assert 0 < t.heads <= BH
    got = sorted(x for c in walk_single(t, BH, T, nsplit, G) for x in c)
    assert got == sorted((bh, h, n) for bh in range(BH) for h in range(nsplit) for n in range(T))


@pytest.mark.parametrize("fwd", [True, False])
@pytest.mark.parametrize("N,wl,wr", [(1000, 1 << 30, 1 << 30), (1000, 1 << 30, 0), (900, 200, 60)])
def test_mask_plan_costs_count_the_computed_blocks(mask_plan, fwd, N, wl, wr):
    """On one head and one CTA per item, the tail runs item b on its own CTA
    when every item fits, longest first; so the table's order gives the
    planner's costs back (strictly, where they differ)."""
    T = -(-N // 128)
    rng = __import__("numpy").random.default_rng(5)
    bm = (rng.random((T, T)) < 0.5).astype("uint8")
    want = mask_costs(bm, fwd, N, wl, wr)
    # a single CTA takes every item of one head in cost order (T <= 8 items)
    t = mask_plan(bm, 1, 1, 1, fwd, N, wl, wr)
    assert t.heads == 1
    order = [e & 2047 for e in t.item[0] if e >= 0]
    assert sorted(order) == list(range(T))
    costs = [want[b] for b in order]
    assert costs == sorted(costs, reverse=True)
    # ties keep block order
    for a, b in zip(order, order[1:]):
        if want[a] == want[b]:
            assert a < b


def test_mask_plan_costs_decide_the_order_on_many_ctas(mask_plan):
    """A mask whose rows (forward) or columns (backward) hold k blocks for
    item k: each item goes to its own CTA, the costliest to CTA 0."""
    import numpy as np
    T = 6
    bm = np.tril(np.ones((T, T), np.uint8))          # row a: a + 1 blocks; column b: T - b
    t = mask_plan(bm, 1, 1, T, True, 128 * T)
    assert [t.item[c][0] & 2047 for c in range(T)] == [5, 4, 3, 2, 1, 0]
    t = mask_plan(bm, 1, 1, T, False, 128 * T)
    assert [t.item[c][0] & 2047 for c in range(T)] == [0, 1, 2, 3, 4, 5]


@pytest.mark.parametrize("BH,nsplit,G,fwd,bound", [
    (32, 1, 152, True, 0.03), (32, 1, 152, False, 0.03), (32, 2, 152, False, 0.03)])
def test_mask_plan_balances_the_block_sparse_step(mask_plan, BH, nsplit, G, fwd, bound):
    """On the local + global + random mask, round-robin leaves the busiest SM
    10 to 35 % above the mean; the planned tail brings it within `bound`."""
    bm = bench_mask()
    T = bm.shape[0]
    cost = mask_costs(bm, fwd, 128 * T, 1 << 30, 1 << 30)
    t = mask_plan(bm, BH, nsplit, G, fwd, 128 * T)
    loads = [sum(cost[n] for _, _, n in c) for c in walk_single(t, BH, T, nsplit, G)]
    mean = sum(loads) / G
    rr = [0] * G
    for u in range(BH * T * nsplit):
        rr[u % G] += cost[(u // nsplit) % T]
    assert max(rr) > mean * 1.1
    assert max(loads) <= mean * (1 + bound), (max(loads) / mean, max(rr) / mean)


def test_mask_plan_without_a_mask_plans_nothing(mask_plan):
    t = TailTable()
    f = getattr(fa.load(), MASK_PLAN)
    f(None, 32, 64, 1, 152, True, 8192, 1 << 30, 1 << 30, 0, ctypes.byref(t))
    assert t.heads == 0
    assert all(t.item[c][k] == -1 for c in range(TAIL_CTAS) for k in range(TAIL_ITEMS))


def test_mask_plans_are_memoised_per_mask(mask_plan):
    """Two masks of one shape get their own plans, and asking again, after
    other plans, returns each one's plan unchanged."""
    import numpy as np
    a = bench_mask(seed=12)
    b = np.ascontiguousarray(a[::-1])                 # the same rows in reverse order
    pa, pb = mask_plan(a, 32, 1, 152, True, 8192), mask_plan(b, 32, 1, 152, True, 8192)
    rows = lambda t: [list(t.item[c]) for c in range(TAIL_CTAS)]
    assert rows(pa) != rows(pb)
    for _ in range(2):
        for s in range(9):                            # more plans than the memo holds
            mask_plan(bench_mask(seed=100 + s), 32, 1, 152, True, 8192)
        assert rows(mask_plan(a, 32, 1, 152, True, 8192)) == rows(pa)
        assert rows(mask_plan(b, 32, 1, 152, True, 8192)) == rows(pb)


@pytest.mark.parametrize("B,H,N,d,fwd", [
    (8, 32, 4096, 128, True), (4, 32, 8192, 128, True), (2, 32, 16384, 128, True),
    (1, 32, 32768, 128, True), (2, 16, 8192, 128, True), (2, 16, 8192, 256, True),
    (2, 16, 8192, 128, False), (2, 16, 8192, 256, False)])
def test_last_head_of_the_large_workloads_runs_in_the_tail(plan, B, H, N, d, fwd):
    """The GPU parity tests of the long-sequence and large-head workloads
    compare every row of four heads, always including the last head
    (B-1, H-1).  With 152 CTAs (one GB300) that head's items run in the
    host-planned tail, with the arguments the launches pass, so the full-size
    parity covers both the paired units and the tail."""
    BH, T = B * H, N // 128
    nsplit = 2 if (not fwd and d == 256) else 1
    head_bytes = 2 * N * d * 2                     # K+V (forward) or Q+dO (backward)
    G = min(BH * T * (1 if fwd else nsplit), 152)
    t = plan(BH, T, nsplit, G, fwd, head_bytes)
    assert t.heads >= 1
    tail_heads = {e >> 12 for c in range(min(G, TAIL_CTAS)) for e in t.item[c] if e >= 0}
    assert BH - 1 in tail_heads
