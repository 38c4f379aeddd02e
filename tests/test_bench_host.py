"""Host logic of the benchmark (no GPU): the counted FLOPs of the sliding-window leg."""

import numpy as np
import pytest

import bench
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A


@pytest.mark.parametrize("N,window,causal", [(300, (37, 0), True), (300, (37, 11), False), (257, (0, 0), False),
                                             (129, (-1, 5), False), (129, (500, 0), True)])
def test_window_pairs_is_the_visible_pair_count(N, window, causal):
    w = inputs.Workload("t", 1, 1, 1, N, N, 64, causal, window=window)
    rows = np.arange(N)
    hidden = A.window_mask(rows, N, *window)
    if causal:
        hidden |= A.causal_mask(rows, N)
    assert bench.window_pairs(w) == int((~hidden).sum())


def test_window_workload_flops():
    w = inputs.WINDOW_N16384_W4096
    # 4096 rows still growing (1 + 2 + ... + 4096 keys), then 12288 rows of 4096 keys
    assert bench.window_pairs(w) == 4096 * 4097 // 2 + 12288 * 4096
    assert bench.fwd_flops(w) == 4.0 * 32 * 128 * bench.window_pairs(w)


def test_window_leg_is_outside_the_step():
    train, dec, win = bench.workloads()
    assert [w.name for w in win] == list(bench.WINDOW)
    assert all(w.window is None for w in train + dec)


def test_varlen_leg_lengths_and_flops():
    w = inputs.VARLEN_T32768_D128
    lens = bench.varlen_lens(w)
    assert len(lens) == 24 and sum(lens) == w.Nq and min(lens) >= 64 and max(lens) <= 8192
    assert lens == inputs.varlen_lengths(24, w.Nq, seed=w.seed)          # seeded: the same every call
    assert bench.fwd_flops(w) == sum(2.0 * w.Hq * n * n * w.d for n in lens)   # causal: half of 4*H*n^2*d


def test_blocksparse_leg_counts_visible_pairs():
    w = inputs.Workload("bs", 1, 2, 2, 1280, 1280, 64, True, extra={"local_tiles": 3, "global_tiles": 1})
    M = np.array(bench.blocksparse_table(w))
    rows = [np.flatnonzero(r) for r in M]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    vis = np.repeat(np.repeat(A.block_mask_from_csr(rp, np.concatenate(rows), 10, 10), 128, 0), 128, 1)
    vis &= ~A.causal_mask(np.arange(1280), 1280)
    assert bench.fwd_flops(w) == 4.0 * 2 * 64 * vis.sum()
    assert M[5].tolist() == [True, False, False, True, True, True, False, False, False, False]


def test_outlier_channel_is_one_per_workload():
    """Every draw of an outlier workload (with or without dO) scales the same channel."""
    w = inputs.Workload("o", 1, 2, 1, 64, 64, 128, True, outliers=True, seed=3)
    a, b = inputs.make(w), inputs.make(w, with_do=False)
    assert a["outlier_channel"] == b["outlier_channel"] == inputs.outlier_channel(128, 3)
    assert int(a["q"].float().abs().mean(dim=(0, 1, 2)).argmax()) == a["outlier_channel"]
    assert inputs.outlier_channel(inputs.GQA_N8192_D128.d, inputs.GQA_N8192_D128.seed) == 44


def test_oracle_sample_flops_count_visible_pairs():
    w = inputs.Workload("c", 1, 1, 1, 300, 300, 64, True)
    rows = np.arange(10, 50)
    assert bench.visible_pairs(w, rows) == int((~A.causal_mask(rows, 300)).sum())
    assert bench.sample_flops(w, "fwd", rows) == 4.0 * 64 * bench.visible_pairs(w, rows)
    assert bench.sample_flops(w, "bwd", rows) == 2.5 * bench.sample_flops(w, "fwd", rows)
    full = inputs.Workload("f", 1, 1, 1, 300, 200, 64, False)
    assert bench.visible_pairs(full, rows) == 40 * 200


def test_training_legs_are_the_benchmark_plan():
    train, dec, _ = bench.workloads()
    assert [w.name for w in train] == ["mha_b4_h16_n2048_d64", "causal_b2_h16_n4096_d128",
                                       "gqa_causal_b1_hq32_hkv8_n8192_d128_outliers"]
    assert bench.tiny_workload() is inputs.TINY
    assert set(bench.TARGET_TRAIN) <= {w.name for w in train}


def test_trace_summary_of_a_synthetic_trace():
    """Two CTAs; CTA 0 runs units 0 and 2, CTA 1 runs unit 1 (times in ns)."""
    t = np.zeros(4096 + 16 * 3, dtype=np.int64)
    t[0:4] = [1000, 11000, 5, 2]
    t[4:8] = [2000, 9000, 7, 1]
    for u, r in enumerate([[1000, 1500, 5000, 6000, 0], [2000, 2500, 8000, 9000, 1], [5000, 6000, 10000, 11000, 0]]):
        t[4096 + 16 * u:4096 + 16 * u + 5] = r
    s = bench.trace_summary(t, 3)
    assert s["ctas"] == 2 and s["span_us"] == 10.0 and s["start_spread_us"] == 1.0
    assert s["busy_us"] == {"min": 7.0, "median": 8.5, "max": 10.0} and s["end_spread_us"] == 2.0
    assert s["units_per_cta"] == {"min": 1.0, "median": 1.5, "max": 2.0}
    assert s["unit_claim_to_first_product_us"]["max"] == 1.0
    assert s["unit_last_product_to_output_us"] == {"min": 1.0, "median": 1.0, "max": 1.0}
    assert s["issue_share_of_busy"] == round((3.5 + 5.5 + 4.0) / 17.0, 4)


def test_forward_launch_count_follows_the_split_plan():
    """A forward call launches the header clear and the forward, plus the combine
    kernel exactly when the shape's key-split plan splits (unmasked shapes only)."""
    import exact_io_aware_21_gb300 as fa
    from exact_io_aware_21_gb300 import binding as B

    lib = fa.library()
    train, dec, win = bench.workloads()
    counts = {}
    for w in train + win + [bench.tiny_workload()]:
        s = B.shape(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.scale, w.causal, w.window)
        counts[w.name] = bench.fwd_kernels(lib, s, 152)
        if w.causal or w.window:
            assert counts[w.name] == 2
    # B4 H16 N2048 d64: 512 units of two query tiles, 56 in the last wave of 152 SMs
    assert counts["mha_b4_h16_n2048_d64"] == 3
    assert counts["tiny_b1_h1_n256_d64"] == 2  # one unit of two key tiles: too short to split
    # the same shape on an SM count that divides its units does not split
    s = B.shape(4, 16, 16, 2048, 2048, 64, 0.125, False)
    assert bench.fwd_kernels(lib, s, 128) == 2
