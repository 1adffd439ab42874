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


def test_roofline_fraction_takes_the_lower_roof():
    """min(pi, AI * beta): a run above the ridge point is measured against the
    dense peak, one below it against the bandwidth roof."""
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 1000.0}   # ridge at 1000 FLOP/B
    # AI = 1e4 FLOP/B: compute roof 1e15 FLOP/s; 1e12 FLOP in 2 ms is half of it
    assert bench.roofline_frac(1e12, 1e8, 2.0, peaks) == 0.5
    # AI = 100 FLOP/B: bandwidth roof 1e14 FLOP/s; 1e12 FLOP in 20 ms is half of it
    assert bench.roofline_frac(1e12, 1e10, 20.0, peaks) == 0.5
    # exactly at the ridge both roofs agree
    assert bench.roofline_frac(1e12, 1e9, 1.0, peaks) == 1.0


def _pairs_brute(N, causal, window, nq=None):
    """Visible (query, key) pairs by enumerating a boolean mask."""
    import numpy as np
    q = np.arange(N)[:, None] if nq is None else (N - nq + np.arange(nq))[:, None]
    k = np.arange(N)[None, :]
    vis = np.ones((q.shape[0], N), dtype=bool)
    if causal:
        vis &= k <= q
    if window is not None:
        wl, wr = window
        if wl >= 0:
            vis &= k >= q - wl
        if wr >= 0:
            vis &= k <= q + wr
    return int(vis.sum())


def test_workload_flop_counts_against_a_mask():
    """The FLOP convention 4 d per visible pair (N^2, N^2 / 2 causal, the
    exact count under a window, decode queries at the end of the cache)."""
    from exact_attention_04_gb300.workloads import Workload
    for N in (1, 7, 128, 300):
        for causal in (False, True):
            for window in (None, (0, 0), (3, -1), (-1, 5), (17, 2)):
                w = Workload("t", 2, 3, N, 64, causal=causal, seed=0, backward=True, window=window)
                brute = _pairs_brute(N, causal, window)
                if window is None and causal:
                    assert w.visible_pairs() == N * N / 2      # the headline convention
                else:
                    assert w.visible_pairs() == brute, (N, causal, window)
                assert w.fwd_flops() == 4.0 * 2 * 3 * 64 * w.visible_pairs()
                assert w.bwd_flops() == 2.5 * w.fwd_flops()
            for nq in (1, 4):
                if nq > N:
                    continue
                w = Workload("t", 1, 1, N, 64, causal=causal, seed=0, backward=False, nq=nq,
                             window=(5, 0))
                assert w.visible_pairs() == _pairs_brute(N, causal, (5, 0), nq=nq)


def test_committed_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """A committed DRAM figure is reported only while every source it depends
    on is unchanged (a stale capture reads as null)."""
    import json
    csrc = tmp_path / "exact_attention_04_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES["bwd_dt_kernel"]:
        (csrc / name).write_text(f"// {name}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    entry = {"kernel": "bwd_dt_kernel", "workload": "w", "dram_bytes_per_launch": 123,
             "source_sha": bench.source_sha("bwd_dt_kernel")}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps([entry]))
    assert bench.committed_traffic("bwd_dt_kernel", "w") == 123
    assert bench.committed_traffic("bwd_dt_kernel", "other") is None
    assert bench.committed_traffic("fa_fwd_kernel", "w") is None
    # any shared header counts, not only the kernel's own file
    (csrc / "sm103_ptx.cuh").write_text("// changed\n")
    assert bench.committed_traffic("bwd_dt_kernel", "w") is None


def test_block_sparse_mask_pattern():
    """Local band, global rows and columns and seeded random blocks, about a
    quarter of the blocks at T = 64, the same mask for the same seed."""
    import numpy as np
    from exact_attention_04_gb300.workloads import block_sparse_mask
    for seed in (0, 1, 2):
        bm = block_sparse_mask(64, seed=seed)
        assert bm.shape == (64, 64) and bm.dtype == np.uint8
        assert np.array_equal(bm, block_sparse_mask(64, seed=seed))
        a, b = np.indices(bm.shape)
        assert bm[np.abs(a - b) <= 4].all()          # local band
        assert bm[:, :2].all() and bm[:2, :].all()   # global key and query blocks
        rows = bm[2:].sum(axis=1)
        assert (rows >= 9).all() and (rows <= 9 + 2 + 5).all()
        assert 0.2 < bm.mean() < 0.3
    assert not np.array_equal(block_sparse_mask(64, seed=0), block_sparse_mask(64, seed=1))


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference times the fp64 oracle on the host cores and
    prints the one JSON line of the contract, with its own cpu_baseline and an
    e2e that moves no bytes."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "single_head_b1_h1_n256_d64", "--steps", "2", "--warmup", "1"],
                         cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC
    assert r["unit"] == "TFLOP/s" and r["value"] > 0 and r["higher_is_better"] is True
    assert (r["n_gpus"], r["steps"], r["warmup"]) == (1, 2, 1)
    assert r["config"]["workload"] == "single_head_b1_h1_n256_d64"
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["cores"] >= 1
    assert r["cpu_baseline"]["value"] == r["value"]
    assert r["e2e"] == {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert r["vs_baseline"] is None


def test_cpu_baseline_extrapolates_from_its_head_sample():
    """The oracle baseline times one head and states the whole workload's
    extrapolated time, B*H times the sample's, next to the small configs run
    whole."""
    from exact_attention_04_gb300.workloads import random_case, make_inputs
    w = random_case(3, 2, 256, 64, seed=5, causal=True)
    cb = bench.cpu_baseline(w, make_inputs(w))
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s" and cb["value"] > 0
    assert cb["extrapolated"]["heads"] == 6
    assert abs(cb["extrapolated"]["seconds"] - 6 * cb["seconds"]) <= 6e-3
    assert [c["workload"] for c in cb["whole_small_configs"]] == list(bench.ORACLE_WHOLE)
