"""Pins of the oracle's block-sparse attention (no GPU).

Against: dense and causal attention (every block listed), attention of each
query block over the gathered keys of its listed blocks (a different route to
the same numbers), the sliding-window oracle where the window is block
aligned, rows that see no key, and rejection of malformed tables.
"""

import numpy as np
import pytest

from oracle import attention as A

RNG = np.random.default_rng(31)


def csr(M):
    rows = [np.flatnonzero(r) for r in M]
    row_ptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    col_idx = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)
    return row_ptr, col_idx


def qkv(B, Hq, Hkv, Nq, Nk, d):
    return (RNG.standard_normal((B, Nq, Hq, d)), RNG.standard_normal((B, Nk, Hkv, d)),
            RNG.standard_normal((B, Nk, Hkv, d)))


@pytest.mark.parametrize("causal", [False, True])
def test_all_blocks_listed_is_dense(causal):
    q, k, v = qkv(2, 2, 1, 40, 40, 8)
    rp, ci = csr(np.ones((5, 5), bool))
    O, L = A.attention_blocksparse_forward(q, k, v, rp, ci, 0.3, causal, block=8)
    Od, Ld = A.attention_forward(q, k, v, 0.3, causal)
    assert np.allclose(O, Od, atol=1e-13) and np.allclose(L, Ld, atol=1e-13)


def test_each_query_block_is_attention_over_its_gathered_keys():
    block, nqb, nkb = 8, 4, 6
    q, k, v = qkv(1, 3, 3, nqb * block - 3, nkb * block - 5, 4)   # ragged last blocks
    M = RNG.random((nqb, nkb)) < 0.5
    M[np.arange(nqb), RNG.integers(0, nkb, nqb)] = True          # every row lists something
    rp, ci = csr(M)
    O, L = A.attention_blocksparse_forward(q, k, v, rp, ci, 0.7, block=block)
    for i in range(nqb):
        rows = np.arange(i * block, min(q.shape[1], (i + 1) * block))
        keys = np.concatenate([np.arange(j * block, min(k.shape[1], (j + 1) * block)) for j in np.flatnonzero(M[i])])
        Og, Lg = A.attention_forward(q[:, rows], k[:, keys], v[:, keys], 0.7)
        assert np.allclose(O[:, rows], Og, atol=1e-13) and np.allclose(L[:, :, rows], Lg, atol=1e-13)


def test_block_tridiagonal_is_a_block_aligned_window():
    block, nb = 8, 6
    q, k, v = qkv(1, 2, 2, nb * block, nb * block, 4)
    M = np.abs(np.subtract.outer(np.arange(nb), np.arange(nb))) <= 1
    rp, ci = csr(M)
    O, L = A.attention_blocksparse_forward(q, k, v, rp, ci, 0.5, block=block)
    # row i sees keys of blocks i//8 - 1 .. i//8 + 1, i.e. the window [8*(i//8) - 8, 8*(i//8) + 15]
    for i in (0, 13, 47):
        lo, hi = max(0, 8 * (i // 8) - 8), min(nb * block - 1, 8 * (i // 8) + 15)
        Ow, Lw = A.attention_forward(q[:, [i]], k[:, lo:hi + 1], v[:, lo:hi + 1], 0.5)
        assert np.allclose(O[:, [i]], Ow, atol=1e-13) and np.allclose(L[:, :, [i]], Lw, atol=1e-13)


def test_rows_that_see_no_key():
    q, k, v = qkv(1, 1, 1, 24, 24, 4)
    M = np.zeros((3, 3), bool)
    M[1, 2] = True                                               # block 1 sees only keys above it
    rp, ci = csr(M)
    O, L = A.attention_blocksparse_forward(q, k, v, rp, ci, 1.0, causal=True, block=8)
    assert np.all(O == 0) and np.all(np.isneginf(L))            # causal hides the only listed block
    O2, L2 = A.attention_blocksparse_forward(q, k, v, rp, ci, 1.0, block=8)
    assert np.all(O2[:, :8] == 0) and np.all(np.isfinite(L2[:, :, 8:16]))


@pytest.mark.parametrize("rp,ci", [([0, 2, 3], [1, 1, 0]), ([0, 2, 3], [1, 0, 0]), ([0, 1, 2], [0, 3]),
                                   ([0, 1], [0])])
def test_malformed_tables_rejected(rp, ci):
    q, k, v = qkv(1, 1, 1, 16, 24, 4)
    with pytest.raises(ValueError):
        A.attention_blocksparse_forward(q, k, v, rp, ci, 1.0, block=8)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_all_blocks_listed_is_dense(causal):
    q, k, v = qkv(1, 2, 1, 40, 40, 8)
    do = RNG.standard_normal(q.shape)
    rp, ci = csr(np.ones((5, 5), bool))
    g = A.attention_blocksparse_backward(q, k, v, do, rp, ci, 0.3, causal, block=8)
    gd = A.attention_backward(q, k, v, do, 0.3, causal)
    for a, b in zip(g, gd):
        assert np.allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_central_differences(causal):
    block, nb = 4, 4
    q, k, v = qkv(1, 2, 1, nb * block - 1, nb * block - 1, 3)
    M = RNG.random((nb, nb)) < 0.5
    M[np.arange(nb), np.arange(nb)] = True
    M[2] = False                                                 # a query block that sees nothing
    rp, ci = csr(M)
    W = RNG.standard_normal(q.shape)
    dq, dk, dv = A.attention_blocksparse_backward(q, k, v, W, rp, ci, 0.6, causal, block=block)
    assert not dq[0, 8:12].any()

    def loss(q_, k_, v_):
        return np.sum(A.attention_blocksparse_forward(q_, k_, v_, rp, ci, 0.6, causal, block=block)[0] * W)

    eps = 1e-6
    for name, x, gr in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, x.shape[1] - 1, x.shape[2] - 1, 2), (0, 6, 0, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            am = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num = (loss(*ap) - loss(*am)) / (2 * eps)
            assert abs(num - gr[idx]) < 1e-6 * max(1.0, abs(num)), (name, idx, num, gr[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sampled_equals_the_full_backward(causal):
    """The per-block sampled backward gives the full backward's rows (head by head;
    dK, dV as one head's contributions, summed over the group)."""
    block, nb = 4, 5
    N = nb * block - 2
    q, k, v = qkv(2, 4, 2, N, N, 3)
    do = RNG.standard_normal(q.shape)
    M = RNG.random((nb, nb)) < 0.5
    M[np.arange(nb), 0] = True
    M[3] = False
    rp, ci = csr(M)
    dq, dk, dv = A.attention_blocksparse_backward(q, k, v, do, rp, ci, 0.4, causal, block=block)
    q_rows, k_rows = np.array([0, 5, 13, N - 1]), np.array([0, 3, 9, N - 1])
    for b in range(2):
        for kvh in range(2):
            sk, sv = np.zeros((4, 3)), np.zeros((4, 3))
            for h in (2 * kvh, 2 * kvh + 1):
                rq, rk, rv = A.attention_blocksparse_backward_sampled(q, k, v, do, rp, ci, 0.4, causal, b, h,
                                                                      q_rows, k_rows, block=block)
                assert np.allclose(rq, dq[b, q_rows, h], atol=1e-12)
                sk += rk
                sv += rv
            assert np.allclose(sk, dk[b, k_rows, kvh], atol=1e-12)
            assert np.allclose(sv, dv[b, k_rows, kvh], atol=1e-12)
