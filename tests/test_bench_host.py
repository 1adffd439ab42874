"""Host-side helpers of bench.py (no GPU needed)."""
import itertools

import bench


def test_visible_pairs_against_brute_force():
    """The useful-FLOPs figure of a padded workload counts the (query, key)
    pairs that key padding (and the causal mask) leave visible."""
    for N, L, causal in itertools.product((1, 5, 17, 64), (0, 1, 3, 17, 64, 80), (False, True)):
        brute = sum(1 for i in range(N) for j in range(N)
                    if j < min(L, N) and (not causal or j <= i))
        assert bench.visible_pairs(L, N, causal) == brute, (N, L, causal)
