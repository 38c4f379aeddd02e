"""Pins of the oracle's FlashDecoding combine and of its integer plans."""

import json
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import plan as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(7)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


@pytest.mark.parametrize("Nk,S", [(1000, 3), (1000, 8), (300, 8), (128, 1), (129, 2), (5000, 19)])
def test_split_then_combine_equals_unsplit(Nk, S):
    """§18.8.2: combining per-split (m_t, l_t, O_t) reproduces attention over all keys."""
    q, k, v = rand(2, 4, 8, 16, scale=2), rand(2, Nk, 2, 16), rand(2, Nk, 2, 16)
    splits = P.decode_splits(Nk, S)
    m, l, Ot = A.decode_partials(q, k, v, 0.25, splits)
    O, L = A.decode_combine(m, l, Ot)
    Of, Lf = A.attention_forward(q, k, v, 0.25)
    np.testing.assert_allclose(O, Of.transpose(0, 2, 1, 3), atol=1e-12)
    np.testing.assert_allclose(L, Lf, atol=1e-12)


def test_partial_is_attention_over_its_keys():
    q, k, v = rand(1, 1, 4, 8), rand(1, 600, 2, 8), rand(1, 600, 2, 8)
    splits = [(0, 256), (256, 600)]
    m, l, Ot = A.decode_partials(q, k, v, 0.4, splits)
    O1, L1 = A.attention_forward(q, k[:, 256:600], v[:, 256:600], 0.4)
    np.testing.assert_allclose(Ot[..., 1, :] / l[..., 1, None], O1.transpose(0, 2, 1, 3), atol=1e-13)
    np.testing.assert_allclose(m[..., 1] + np.log(l[..., 1]), L1, atol=1e-13)


def test_empty_split_has_zero_weight():
    q, k, v = rand(1, 1, 2, 8), rand(1, 64, 1, 8), rand(1, 64, 1, 8)
    m, l, Ot = A.decode_partials(q, k, v, 0.4, [(0, 64), (64, 64)])
    assert np.all(np.isneginf(m[..., 1])) and not l[..., 1].any()
    O, L = A.decode_combine(m, l, Ot)
    Of, Lf = A.attention_forward(q, k, v, 0.4)
    np.testing.assert_allclose(O, Of.transpose(0, 2, 1, 3), atol=1e-13)


@pytest.mark.parametrize("Nk", [1, 127, 128, 129, 1000, 131072])
@pytest.mark.parametrize("S", [1, 2, 7, 19, 64])
def test_decode_splits_partition_the_keys(Nk, S):
    sp = P.decode_splits(Nk, S)
    assert 1 <= len(sp) <= S
    assert sp[0][0] == 0 and sp[-1][1] == Nk
    for (a0, a1), (b0, b1) in zip(sp, sp[1:]):
        assert a1 == b0
    for s0, s1 in sp:
        assert s1 > s0 and s0 % P.TILE == 0
    assert len({s1 - s0 for s0, s1 in sp[:-1]}) <= 1   # equal chunks but the last


def test_lpt_worked_example():
    """Lecture slides 27-46: loads [9, 5, 6] in order, [7, 7, 6] longest first."""
    g = json.load(open(os.path.join(GOLDEN, "lpt_example.json")))
    assert P.greedy_loads(g["jobs_in_order"], g["workers"], False) == g["printed"]["in_order_loads"]
    assert P.greedy_loads(g["jobs_in_order"], g["workers"], True) == g["printed"]["longest_first_loads"]
    # the jobs are the key-tile counts of 2 batches x 4 causal query tiles
    costs = [P.fwd_unit_cost(4 * 128, 4 * 128, True, 0)]  # pair (0, 1) visits 2 tiles
    assert costs == [2]
    per_tile = [sum(1 for c in row if c != P.SKIP) for row in P.tile_classes(512, 512, 128, 128, True)]
    assert per_tile * 2 == g["jobs_in_order"]


def test_causal_figure_3x3():
    """Fig. 18-20: lower triangle and diagonal computed, upper triangle skipped."""
    g = json.load(open(os.path.join(GOLDEN, "causal_blocks_3x3.json")))
    n = g["blocks"]
    cls = P.tile_classes(n * 128, n * 128, 128, 128, True)
    got = [["skip" if c == P.SKIP else "compute" for c in row] for row in cls]
    assert got == g["pattern"]
    assert [cls[i][i] for i in range(n)] == [P.PARTIAL] * n


@pytest.mark.parametrize("N,bm,bn", [(10, 4, 4), (13, 4, 3), (9, 2, 5), (256, 128, 128), (300, 128, 128),
                                     (17, 16, 16)])
def test_tile_classes_match_brute_force(N, bm, bn):
    """Each class equals what the element mask j > i says about the whole block."""
    mask = np.arange(N)[None, :] > np.arange(N)[:, None]
    cls = P.tile_classes(N, N, bm, bn, True)
    for i, row in enumerate(cls):
        for j, c in enumerate(row):
            blk = mask[i * bm:(i + 1) * bm, j * bn:(j + 1) * bn]
            want = P.SKIP if blk.all() else (P.FULL if not blk.any() else P.PARTIAL)
            assert c == want, (i, j)


@pytest.mark.parametrize("N", [128, 200, 256, 1000, 4096])
def test_visited_tiles_match_pages_bound(N):
    """§18.5.2: the causal loop visits ceil((q_start + B_r) / B_c) key tiles (clipped)."""
    cls = P.tile_classes(N, N, 128, 128, True)
    for i, row in enumerate(cls):
        bound = min(P.cdiv(N, 128), P.cdiv(i * 128 + 128, 128))
        assert sum(1 for c in row if c != P.SKIP) == bound
        assert all(c == P.SKIP for c in row[bound:])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 300, 1024])
def test_unit_orders_are_longest_first_permutations(causal, N):
    B, Hq, Hkv = 2, 4, 2
    f = P.fwd_unit_order(B, Hq, N, N, causal)
    assert len(set(f)) == len(f) == B * Hq * P.cdiv(P.cdiv(N, 128), 2)
    costs = [P.fwd_unit_cost(N, N, causal, u[2]) for u in f]
    assert costs == sorted(costs, reverse=True)
    kv = P.dkdv_unit_order(B, Hkv, N, N, causal)
    assert len(set(kv)) == len(kv) == B * Hkv * P.cdiv(N, 128)
    if causal:
        assert [u[2] for u in kv] == sorted(u[2] for u in kv)   # early key tiles see most queries
    dq = P.dq_unit_order(B, Hq, N, N, causal)
    if causal:
        assert [u[2] for u in dq] == sorted((u[2] for u in dq), reverse=True)


def test_lpt_beats_in_order_on_causal_units():
    costs = [P.fwd_unit_cost(4096, 4096, True, p) for p in range(16)] * 32
    a = max(P.greedy_loads(costs, 152, False))
    b = max(P.greedy_loads(costs, 152, True))
    assert b <= a and b <= 1.1 * sum(costs) / 152 + max(costs)
