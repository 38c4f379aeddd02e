"""Pins of the paged, variable-length decode oracle (no GPU).

Each pin ties it to something fixed outside the function: the dense oracle on
the same keys laid out contiguously, closed forms for Q = 0 and for a single
key, invariance under relabelling the physical pages, and isolation from rows
the page table does not reference.
"""

import numpy as np
import pytest

from oracle import attention as A


def paged_layout(k, v, page_size, rng=None, spare=3):
    """Lay contiguous K/V [B, N, H, d] out in pages, optionally shuffled, with spare pages."""
    B, N, H, d = k.shape
    npb = -(-N // page_size)
    pages = B * npb + spare
    order = np.arange(pages) if rng is None else rng.permutation(pages)
    kc = np.full((pages, page_size, H, d), 7.0)   # unreferenced rows hold junk
    vc = np.full((pages, page_size, H, d), -7.0)
    table = np.zeros((B, npb + 2), dtype=np.int64) - 1
    for b in range(B):
        for i in range(npb):
            pg = order[b * npb + i]
            table[b, i] = pg
            rows = slice(i * page_size, min(N, (i + 1) * page_size))
            n = rows.stop - rows.start
            kc[pg, :n] = k[b, rows]
            vc[pg, :n] = v[b, rows]
    return kc, vc, table


def draw(B, Nq, Hq, Hkv, N, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Nq, Hq, d)), rng.standard_normal((B, N, Hkv, d)),
            rng.standard_normal((B, N, Hkv, d)))


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_identity_layout_equals_dense_oracle(page_size):
    q, k, v = draw(2, 4, 8, 2, 300, 16, 1)
    kc, vc, table = paged_layout(k, v, page_size)
    lens = np.array([300, 300])
    O, LSE = A.attention_decode_paged(q, kc, vc, table, lens, 0.25)
    Od, LSEd = A.attention_forward(q, k, v, 0.25)
    assert np.array_equal(O, Od) and np.array_equal(LSE, LSEd)


def test_ragged_lengths_attend_to_their_prefix_only():
    q, k, v = draw(3, 1, 4, 1, 257, 8, 2)
    kc, vc, table = paged_layout(k, v, 32, rng=np.random.default_rng(5))
    lens = np.array([1, 100, 257])
    O, LSE = A.attention_decode_paged(q, kc, vc, table, lens, 0.5)
    for b, L in enumerate(lens):
        Ob, LSEb = A.attention_forward(q[b:b + 1], k[b:b + 1, :L], v[b:b + 1, :L], 0.5)
        assert np.array_equal(O[b], Ob[0]) and np.array_equal(LSE[b], LSEb[0])


def test_relabelling_physical_pages_changes_nothing():
    q, k, v = draw(2, 4, 4, 2, 200, 8, 3)
    lens = np.array([173, 200])
    a = A.attention_decode_paged(q, *paged_layout(k, v, 16), lens, 0.3)
    b = A.attention_decode_paged(q, *paged_layout(k, v, 16, rng=np.random.default_rng(9)), lens, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_zero_query_gives_prefix_mean_and_log_length():
    _, k, v = draw(2, 1, 2, 2, 150, 8, 4)
    q = np.zeros((2, 3, 2, 8))
    kc, vc, table = paged_layout(k, v, 64, rng=np.random.default_rng(1))
    lens = np.array([37, 150])
    O, LSE = A.attention_decode_paged(q, kc, vc, table, lens, 1.0)
    for b, L in enumerate(lens):
        assert np.allclose(O[b], v[b, :L].mean(axis=0)[None], atol=1e-13)   # [Nq, H, d] vs [1, H, d]
        assert np.allclose(LSE[b], np.log(L), atol=1e-13)


def test_single_key_returns_its_value_and_score():
    q, k, v = draw(1, 2, 4, 2, 64, 8, 6)
    kc, vc, table = paged_layout(k, v, 16)
    O, LSE = A.attention_decode_paged(q, kc, vc, table, np.array([1]), 0.7)
    for h in range(4):
        kv = h // 2
        assert np.allclose(O[0, :, h], v[0, 0, kv][None], atol=1e-15)
        assert np.allclose(LSE[0, h], 0.7 * q[0, :, h] @ k[0, 0, kv], atol=1e-13)


def test_unreferenced_rows_and_pages_do_not_matter():
    q, k, v = draw(2, 1, 2, 1, 100, 8, 7)
    kc, vc, table = paged_layout(k, v, 32, rng=np.random.default_rng(2), spare=4)
    lens = np.array([45, 100])
    base = A.attention_decode_paged(q, kc, vc, table, lens, 0.4)
    used = {(int(table[b, r // 32]), r % 32) for b in range(2) for r in range(lens[b])}
    kc2, vc2 = kc.copy(), vc.copy()
    for pg in range(kc.shape[0]):
        for r in range(32):
            if (pg, r) not in used:
                kc2[pg, r] = 1e6
                vc2[pg, r] = np.nan
    other = A.attention_decode_paged(q, kc2, vc2, table, lens, 0.4)
    assert np.array_equal(base[0], other[0]) and np.array_equal(base[1], other[1])


def test_split_partials_over_gathered_rows_combine_to_the_paged_result():
    q, k, v = draw(1, 4, 4, 1, 500, 8, 8)
    kc, vc, table = paged_layout(k, v, 64, rng=np.random.default_rng(3))
    L = 437
    O, LSE = A.attention_decode_paged(q, kc, vc, table, np.array([L]), 0.35)
    kg = A.gather_paged(kc, table, 0, L)[None]
    vg = A.gather_paged(vc, table, 0, L)[None]
    m, l, Ot = A.decode_partials(q, kg, vg, 0.35, [(0, 128), (128, 256), (256, 384), (384, L)])
    Oc, LSEc = A.decode_combine(m, l, Ot)
    assert np.allclose(Oc.transpose(0, 2, 1, 3), O, atol=1e-13)
    assert np.allclose(LSEc, LSE, atol=1e-13)
