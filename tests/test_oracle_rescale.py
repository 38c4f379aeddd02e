"""Pins of the oracle's conditional-rescaling forward (the L21 notes on FA4: an
online-softmax variant that skips most rescalings of O).

The variant keeps a per-row reference that moves only when a block's max passes
it by more than a threshold.  Exactness does not depend on the reference: the
§18.4.2 update (rescale l and O by exp(r_old - r_new)) is an identity for any
reference, so the result must equal the plain definition for every threshold.
What the threshold changes is how often the reference moves and how large the
unnormalised probabilities get (at most 2^threshold), both counted here against
brute-force counts taken from the score matrix itself.
"""

import numpy as np
import pytest

from oracle import attention as A

RNG = np.random.default_rng(2468)


def plain(Q, K, V, scale, causal):
    O, L = A.attention_forward(Q[None, :, None], K[None, :, None], V[None, :, None], scale, causal)
    return O[0, :, 0], L[0, 0]


@pytest.mark.parametrize("threshold", [0.0, 1.0, 4.0, 8.0, 16.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [(1, 1), (5, 3), (32, 16), (64, 64)])
def test_conditional_rescaling_equals_the_plain_definition(threshold, causal, blocks):
    N, d = 130, 16
    Q, K, V = RNG.standard_normal((N, d)) * 2.0, RNG.standard_normal((N, d)), RNG.standard_normal((N, d))
    scale = 1 / np.sqrt(d)
    O_c, L_c, _, p_max = A.tiled_forward_head_conditional(Q, K, V, scale, blocks[0], blocks[1], threshold, causal)
    O, L = plain(Q, K, V, scale, causal)
    np.testing.assert_allclose(O_c, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L_c, L, rtol=0, atol=1e-12)
    assert p_max <= 2.0 ** threshold * (1 + 1e-12)


def record_moves(S, block, tau):
    """Brute force from the score matrix: per row, the blocks (after the first) whose max
    passes the reference by more than tau, the reference being the max that last moved it."""
    n = 0
    for row in S:
        r = -np.inf
        for j0 in range(0, len(row), block):
            mt = row[j0:j0 + block].max()
            if mt > r + tau:
                n += int(np.isfinite(r))
                r = mt
    return n


@pytest.mark.parametrize("threshold", [0.0, 0.5, 2.0, 8.0])
def test_rescaling_count_matches_brute_force(threshold):
    N, d, block = 200, 32, 16
    Q, K, V = RNG.standard_normal((N, d)), RNG.standard_normal((N, d)), RNG.standard_normal((N, d))
    scale = 1 / np.sqrt(d)
    _, _, n, _ = A.tiled_forward_head_conditional(Q, K, V, scale, 40, block, threshold)
    S = scale * Q @ K.T
    assert n == record_moves(S, block, threshold * np.log(2.0))


def test_threshold_eight_skips_most_rescalings():
    """The notes: the FA4 variant skips about 90% of the rescalings.  On the benchmark's
    N(0,1) inputs (scale 1/sqrt(d), 128-key blocks) a threshold of 8 skips every one
    after the first block, while the exact running max moves several times per row."""
    N, d = 2048, 128
    Q, K, V = RNG.standard_normal((N, d)), RNG.standard_normal((N, d)), RNG.standard_normal((N, d))
    rows = slice(N - 256, N)
    scale = 1 / np.sqrt(d)
    _, _, n0, p0 = A.tiled_forward_head_conditional(Q[rows], K, V, scale, 128, 128, 0.0)
    _, _, n8, p8 = A.tiled_forward_head_conditional(Q[rows], K, V, scale, 128, 128, 8.0)
    assert n0 >= 256 and n8 <= 0.1 * n0
    assert p0 == 1.0 and 1.0 <= p8 <= 256.0


def test_a_late_dominant_key_moves_the_reference_once():
    """A key whose score passes every earlier one by far more than the threshold forces
    exactly one move in each row that sees it, and the output is that key's value."""
    N, d = 64, 8
    Q = np.zeros((N, d))
    Q[:, 0] = 1.0
    K = RNG.standard_normal((N, d)) * 0.01
    K[50, 0] = 80.0           # score 80 / sqrt(8) = 28.3 nats = 40.8 bits above the rest
    V = RNG.standard_normal((N, d))
    O, L, n, _ = A.tiled_forward_head_conditional(Q, K, V, 1 / np.sqrt(d), 64, 8, 8.0)
    assert n == N
    np.testing.assert_allclose(O, np.broadcast_to(V[50], O.shape), rtol=0, atol=1e-5)
    O_ref, L_ref = plain(Q, K, V, 1 / np.sqrt(d), False)
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
