"""Pins of the oracle's forward pass against facts fixed outside the oracle.

Each test would fail for a plausible slip in ``oracle.attention``: a dropped
max subtraction, a wrong scale placement, a transposed operand, a wrong causal
direction, a wrong GQA head mapping, or a wrong log-sum-exp.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def test_two_block_rescaling_identity():
    """Lecture slide 12: O(2) = (l1/l2) O(1) + A2 V2 / l2 equals the one-shot output."""
    d = 16
    Q, K, V = rand(7, d, scale=0.3), rand(20, d, scale=0.3), rand(20, d)
    scale = 1 / np.sqrt(d)
    O2 = A.two_block_output(Q, K[:9], V[:9], K[9:], V[9:], scale)
    O, _ = A.attention_forward(Q[None, :, None], K[None, :, None], V[None, :, None], scale)
    np.testing.assert_allclose(O2, O[0, :, 0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [(1, 1), (3, 5), (16, 7), (64, 64), (128, 128)])
def test_online_softmax_theorem(causal, blocks):
    """§18.4.2 theorem: any blocking of the online recurrence gives the one-shot result."""
    N, d = 150, 24
    Q, K, V = rand(N, d), rand(N, d), rand(N, d)
    scale = 1 / np.sqrt(d)
    O_t, L_t = A.tiled_forward_head(Q, K, V, scale, blocks[0], blocks[1], causal=causal)
    O, L = A.attention_forward(Q[None, :, None], K[None, :, None], V[None, :, None], scale, causal)
    np.testing.assert_allclose(O_t, O[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L_t, L[0, 0], rtol=0, atol=1e-12)


def test_softmax_rows_are_distributions():
    """§18.2.1: softmax entries are positive and each row sums to 1; order is kept."""
    S = rand(9, 33, scale=5.0)
    P, m, l = A._softmax_rows(S)
    assert np.all(P > 0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.array_equal(np.argsort(P, axis=1), np.argsort(S, axis=1))
    np.testing.assert_array_equal(m, S.max(axis=1))


def test_large_scores_do_not_overflow():
    """Safe softmax (§18.4.2): scores near 1e4 still give finite, exact results."""
    d = 8
    Q = np.zeros((1, 3, 1, d))
    Q[0, :, 0, 0] = 1e4
    K = np.zeros((1, 2, 1, d))
    K[0, 0, 0, 0] = 1.0
    K[0, 1, 0, 0] = 1.0 - 1e-4
    V = rand(1, 2, 1, d)
    O, L = A.attention_forward(Q, K, V, 1.0)
    w = 1 / (1 + np.exp(-1.0))  # softmax of (1e4, 1e4 - 1)
    np.testing.assert_allclose(O[0, 0, 0], w * V[0, 0, 0] + (1 - w) * V[0, 1, 0], atol=1e-12)
    np.testing.assert_allclose(L[0, 0, 0], 1e4 + np.log(1 + np.exp(-1.0)), rtol=1e-15)


@pytest.mark.parametrize("Nk", [1, 5, 256])
def test_zero_query_gives_mean_of_values(Nk):
    """Q = 0: every score is 0, so O = mean(V) and LSE = ln Nk (non-causal)."""
    d = 16
    q = np.zeros((2, 4, 2, d))
    k, v = rand(2, Nk, 1, d), rand(2, Nk, 1, d)
    O, L = A.attention_forward(q, k, v, 0.25)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape), atol=1e-14)
    np.testing.assert_allclose(L, np.log(Nk), atol=1e-14)


def test_zero_query_causal_prefix_means():
    """Causal, Q = 0: O_i = mean(V[0..i]) and LSE_i = ln(i + 1) exactly."""
    N, d = 37, 8
    q = np.zeros((1, N, 1, d))
    k, v = rand(1, N, 1, d), rand(1, N, 1, d)
    O, L = A.attention_forward(q, k, v, 1.0, causal=True)
    prefix = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(O[0, :, 0], prefix, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.log(np.arange(1, N + 1)), atol=1e-14)


def test_constant_values_give_constant_output():
    """Every V row equal to c: O = c whatever the scores."""
    d = 12
    q, k = rand(1, 9, 3, d, scale=3), rand(1, 40, 3, d, scale=3)
    c = rand(d)
    v = np.broadcast_to(c, (1, 40, 3, d)).copy()
    for causal in (False,):
        O, _ = A.attention_forward(q, k, v, 0.7, causal)
        np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-13)
    qc, kc = rand(1, 40, 3, d, scale=3), rand(1, 40, 3, d, scale=3)
    O, _ = A.attention_forward(qc, kc, v, 0.7, True)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-13)


def test_causal_row_zero_sees_only_key_zero():
    """Causal row 0: O_0 = V_0 and LSE_0 = scale * q_0 . k_0."""
    d = 16
    q, k, v = rand(2, 10, 2, d), rand(2, 10, 2, d), rand(2, 10, 2, d)
    O, L = A.attention_forward(q, k, v, 0.3, causal=True)
    np.testing.assert_allclose(O[:, 0], v[:, 0], atol=1e-14)
    np.testing.assert_allclose(L[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), atol=1e-13)


def test_two_keys_closed_form():
    """Two keys: softmax is a logistic function of the score difference."""
    d = 6
    q, k, v = rand(1, 3, 1, d), rand(1, 2, 1, d), rand(1, 2, 1, d)
    scale = 0.37
    O, L = A.attention_forward(q, k, v, scale)
    s = scale * q[0, :, 0] @ k[0, :, 0].T          # [3, 2]
    w0 = 1 / (1 + np.exp(s[:, 1] - s[:, 0]))
    np.testing.assert_allclose(O[0, :, 0], w0[:, None] * v[0, 0, 0] + (1 - w0)[:, None] * v[0, 1, 0], atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.logaddexp(s[:, 0], s[:, 1]), atol=1e-14)


def test_key_permutation_invariance():
    """Non-causal attention does not depend on the order of the (key, value) pairs."""
    d = 8
    q, k, v = rand(1, 6, 2, d), rand(1, 30, 2, d), rand(1, 30, 2, d)
    perm = RNG.permutation(30)
    O1, L1 = A.attention_forward(q, k, v, 0.5)
    O2, L2 = A.attention_forward(q, k[:, perm], v[:, perm], 0.5)
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    """Grouped heads (§18.2.2): query head h uses KV head h // g; g = 1 is plain MHA."""
    d, g = 8, 3
    q, k, v = rand(2, 11, 6, d), rand(2, 13, 2, d), rand(2, 13, 2, d)
    O, L = A.attention_forward(q, k, v, 0.4)
    kr, vr = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    O2, L2 = A.attention_forward(q, kr, vr, 0.4)
    np.testing.assert_allclose(O, O2, atol=1e-14)
    np.testing.assert_allclose(L, L2, atol=1e-14)
    # the mapping is consecutive: heads 0..2 -> KV 0, heads 3..5 -> KV 1
    O3, _ = A.attention_forward(q[:, :, 3:4], k[:, :, 1:2], v[:, :, 1:2], 0.4)
    np.testing.assert_allclose(O[:, :, 3:4], O3, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_library_sdpa_in_fp64(causal):
    """Cross-check with PyTorch's math SDPA in float64 (an independent implementation)."""
    B, N, H, d = 2, 45, 3, 16
    q, k, v = rand(B, N, H, d), rand(B, N, H, d), rand(B, N, H, d)
    O, L = A.attention_forward(q, k, v, 0.21, causal)
    t = lambda x: torch.from_numpy(x).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal, scale=0.21)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), atol=1e-13)
    S = torch.einsum("bhid,bhjd->bhij", t(q), t(k)) * 0.21
    if causal:
        S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(L, torch.logsumexp(S, dim=-1).numpy(), atol=1e-13)


def test_row_restriction_matches_full():
    d = 8
    q, k, v = rand(1, 50, 2, d), rand(1, 50, 2, d), rand(1, 50, 2, d)
    O, L = A.attention_forward(q, k, v, 0.3, True)
    rows = np.array([0, 7, 49])
    Os, Ls = A.attention_forward(q, k, v, 0.3, True, heads=[(0, 1)], rows=rows)
    np.testing.assert_allclose(Os[0, rows, 1], O[0, rows, 1], atol=1e-15)
    np.testing.assert_allclose(Ls[0, 1, rows], L[0, 1, rows], atol=1e-15)
    assert np.isnan(Os[0, 1, 1]).all() and np.isnan(Os[0, 0, 0]).all()


def test_flop_count_closed_forms():
    """§18.2.3: about 4 N^2 d per head; §18.5.2: causal is half, 2 N^2 d."""
    assert A.flops_forward(1, 1, 100, 100, 8, False) == 4 * 100 * 100 * 8
    assert A.flops_forward(1, 1, 100, 100, 8, True) == 2 * 100 * 100 * 8
    assert A.flops_forward(4, 16, 2048, 2048, 64, False) == pytest.approx(68.72e9, rel=1e-3)
    assert A.flops_backward(2, 16, 4096, 4096, 128, True) == pytest.approx(343.6e9, rel=1e-3)
