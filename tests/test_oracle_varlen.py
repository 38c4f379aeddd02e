"""Pins of the oracle's packed variable-length attention (no GPU).

Against: the whole packed batch as one attention problem with a block-diagonal
mask (every token attends only within its own sequence), the dense oracle on
one sequence, invariance under reordering the sequences, empty sequences, and
central differences of the packed backward.
"""

import numpy as np
import pytest

from oracle import attention as A

RNG = np.random.default_rng(21)


def packed(lens_q, lens_k, Hq, Hkv, d):
    tq, tk = sum(lens_q), sum(lens_k)
    q, k, v = RNG.standard_normal((tq, Hq, d)), RNG.standard_normal((tk, Hkv, d)), RNG.standard_normal((tk, Hkv, d))
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    return q, k, v, cq, ck


def block_diagonal(q, k, v, cq, ck, scale, causal):
    """All tokens at once: key j is visible to query i iff both lie in the same
    sequence (and, causal, j's position in it is at most i's)."""
    seq_q = np.searchsorted(cq, np.arange(q.shape[0]), side="right") - 1
    seq_k = np.searchsorted(ck, np.arange(k.shape[0]), side="right") - 1
    pos_q = np.arange(q.shape[0]) - cq[seq_q]
    pos_k = np.arange(k.shape[0]) - ck[seq_k]
    vis = seq_q[:, None] == seq_k[None, :]
    if causal:
        vis &= pos_k[None, :] <= pos_q[:, None]
    g = q.shape[1] // k.shape[1]
    O = np.zeros(q.shape)
    L = np.zeros((q.shape[1], q.shape[0]))
    for h in range(q.shape[1]):
        S = np.where(vis, scale * q[:, h] @ k[:, h // g].T, -np.inf)
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        O[:, h] = E @ v[:, h // g] / E.sum(axis=1, keepdims=True)
        L[h] = m[:, 0] + np.log(E.sum(axis=1))
    return O, L


@pytest.mark.parametrize("lens_q,lens_k,causal", [([5, 17, 1, 9], [5, 17, 1, 9], True),
                                                  ([5, 17, 1, 9], [12, 3, 8, 20], False),
                                                  ([33], [33], True)])
def test_packed_equals_block_diagonal_attention(lens_q, lens_k, causal):
    q, k, v, cq, ck = packed(lens_q, lens_k, 4, 2, 8)
    O, L = A.attention_varlen_forward(q, k, v, cq, ck, 0.4, causal)
    Ob, Lb = block_diagonal(q, k, v, cq, ck, 0.4, causal)
    assert np.allclose(O, Ob, atol=1e-12) and np.allclose(L, Lb, atol=1e-12)


def test_one_sequence_is_the_dense_forward():
    q, k, v, cq, ck = packed([40], [40], 2, 1, 8)
    O, L = A.attention_varlen_forward(q, k, v, cq, ck, 0.3, True)
    Od, Ld = A.attention_forward(q[None], k[None], v[None], 0.3, True)
    assert np.array_equal(O, Od[0]) and np.array_equal(L, Ld[0])


def test_reordering_sequences_reorders_outputs_and_empty_ones_are_skipped():
    lens = [7, 0, 12, 3]
    q, k, v, cq, ck = packed(lens, lens, 2, 2, 4)
    O, L = A.attention_varlen_forward(q, k, v, cq, ck, 0.5, True)
    order = [2, 3, 0, 1]                                       # move the sequences around
    pieces = [np.arange(cq[b], cq[b + 1]) for b in order]
    idx = np.concatenate(pieces)
    cq2 = np.concatenate([[0], np.cumsum([lens[b] for b in order])])
    O2, L2 = A.attention_varlen_forward(q[idx], k[idx], v[idx], cq2, cq2, 0.5, True)
    assert np.allclose(O2, O[idx], atol=1e-13) and np.allclose(L2, L[:, idx], atol=1e-13)
    nz = [b for b in range(len(lens)) if lens[b]]              # dropping the empty one changes nothing
    cq3 = np.concatenate([[0], np.cumsum([lens[b] for b in nz])])
    O3, _ = A.attention_varlen_forward(q, k, v, cq3, cq3, 0.5, True)
    assert np.array_equal(O3, O)


def test_causal_needs_equal_lengths():
    q, k, v, cq, ck = packed([4, 6], [6, 4], 1, 1, 4)
    with pytest.raises(ValueError):
        A.attention_varlen_forward(q, k, v, cq, ck, 1.0, True)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_central_differences(causal):
    lens_q = [3, 0, 4] if not causal else [3, 4]
    lens_k = [2, 3, 5] if not causal else [3, 4]
    q, k, v, cq, ck = packed(lens_q, lens_k, 2, 1, 3)
    W = RNG.standard_normal(q.shape)                           # loss = sum(O * W), so dO = W
    dq, dk, dv = A.attention_varlen_backward(q, k, v, W, cq, ck, 0.7, causal)
    if not causal:                                             # sequence 1 has keys but no queries
        assert not dk[ck[1]:ck[2]].any() and not dv[ck[1]:ck[2]].any()

    def loss(q_, k_, v_):
        return np.sum(A.attention_varlen_forward(q_, k_, v_, cq, ck, 0.7, causal)[0] * W)

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0), (x.shape[0] - 1, x.shape[1] - 1, 2), (x.shape[0] // 2, 0, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(num - g[idx]) < 1e-6 * max(1.0, abs(num)), (name, idx, num, g[idx])
