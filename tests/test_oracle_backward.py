"""Pins of the oracle's backward pass: finite differences, autograd, invariants."""

import numpy as np
import pytest
import torch

from oracle import attention as A

RNG = np.random.default_rng(99)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def loss(q, k, v, do, scale, causal):
    O, _ = A.attention_forward(q, k, v, scale, causal)
    return float(np.sum(O * do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("heads", [(2, 2), (2, 1)])
def test_finite_differences(causal, heads):
    """Central differences of L = sum(O * dO) in fp64 match dQ, dK, dV (rel err < 1e-7)."""
    Hq, Hkv = heads
    B, N, d = 1, 7, 4
    scale = 0.6
    q, k, v, do = rand(B, N, Hq, d), rand(B, N, Hkv, d), rand(B, N, Hkv, d), rand(B, N, Hq, d)
    dq, dk, dv = A.attention_backward(q, k, v, do, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = loss(args["q"], args["k"], args["v"], do, scale, causal)
            args[name] = xm
            fm = loss(args["q"], args["k"], args["v"], do, scale, causal)
            num[idx] = (fp - fm) / (2 * h)
        err = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd_fp64(causal):
    """Gradients equal those of PyTorch autograd through a plain fp64 formula."""
    B, N, Hq, Hkv, d = 2, 33, 4, 2, 8
    scale = 0.35
    q, k, v, do = rand(B, N, Hq, d), rand(B, N, Hkv, d), rand(B, N, Hkv, d), rand(B, N, Hq, d)
    dq, dk, dv = A.attention_backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    g = Hq // Hkv
    kk = tk.repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    vv = tv.repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(tq.permute(0, 2, 1, 3), kk, vv,
                                                         is_causal=causal, scale=scale)
    o.permute(0, 2, 1, 3).backward(torch.tensor(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_key_gradients_sum_to_zero():
    """Softmax rows are shift-invariant, so sum_j dS_ij = 0 and sum_j dK_j = 0 (per head)."""
    q, k, v, do = rand(1, 20, 2, 8), rand(1, 25, 2, 8), rand(1, 25, 2, 8), rand(1, 20, 2, 8)
    _, dk, _ = A.attention_backward(q, k, v, do, 0.5, False)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)


def test_zero_upstream_gradient():
    q, k, v = rand(1, 9, 2, 4), rand(1, 9, 2, 4), rand(1, 9, 2, 4)
    dq, dk, dv = A.attention_backward(q, k, v, np.zeros_like(q), 0.5, True)
    assert not dq.any() and not dk.any() and not dv.any()


def test_constant_values_kill_query_and_key_gradients():
    """All V rows = c: dP_ij = dO_i.c = D_i, so dS = 0, dQ = dK = 0, dV_j = sum_i P_ij dO_i."""
    B, N, d = 1, 15, 6
    c = rand(d)
    q, k, do = rand(B, N, 1, d), rand(B, N, 1, d), rand(B, N, 1, d)
    v = np.broadcast_to(c, (B, N, 1, d)).copy()
    dq, dk, dv = A.attention_backward(q, k, v, do, 0.8, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    S = 0.8 * q[0, :, 0] @ k[0, :, 0].T
    P = np.exp(S - S.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    np.testing.assert_allclose(dv[0, :, 0], P.T @ do[0, :, 0], atol=1e-13)


def test_gqa_key_gradient_is_sum_over_group():
    """dK/dV of a shared KV head equal the sum of the per-head MHA gradients."""
    q, k, v, do = rand(1, 10, 4, 8), rand(1, 12, 2, 8), rand(1, 12, 2, 8), rand(1, 10, 4, 8)
    dq, dk, dv = A.attention_backward(q, k, v, do, 0.3, False)
    kr, vr = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    dq2, dk2, dv2 = A.attention_backward(q, kr, vr, do, 0.3, False)
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk, dk2[:, :, 0::2] + dk2[:, :, 1::2], atol=1e-13)
    np.testing.assert_allclose(dv, dv2[:, :, 0::2] + dv2[:, :, 1::2], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_backward_matches_full(causal):
    q, k, v, do = rand(1, 70, 4, 8), rand(1, 70, 2, 8), rand(1, 70, 2, 8), rand(1, 70, 4, 8)
    dq, _, _ = A.attention_backward(q, k, v, do, 0.3, causal)
    _, dk1, dv1 = A.attention_backward(q, k, v, do, 0.3, causal, heads=[(0, 3)])
    qr, kr = np.array([0, 5, 69]), np.array([1, 33, 68])
    sq, sk, sv = A.attention_backward_sampled(q, k, v, do, 0.3, causal, 0, 3, qr, kr, row_block=16)
    np.testing.assert_allclose(sq, dq[0, qr, 3], atol=1e-13)
    np.testing.assert_allclose(sk, dk1[0, kr, 1], atol=1e-13)
    np.testing.assert_allclose(sv, dv1[0, kr, 1], atol=1e-13)


def test_row_block_does_not_change_result():
    q, k, v, do = rand(1, 50, 2, 8), rand(1, 50, 2, 8), rand(1, 50, 2, 8), rand(1, 50, 2, 8)
    a = A.attention_backward(q, k, v, do, 0.3, True, row_block=7)
    b = A.attention_backward(q, k, v, do, 0.3, True, row_block=1000)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13)


def test_row_restriction_sums_to_full():
    """dK, dV are sums over query rows: two disjoint row sets add up to the full result."""
    q, k, v, do = rand(1, 40, 2, 8), rand(1, 40, 1, 8), rand(1, 40, 1, 8), rand(1, 40, 2, 8)
    full = A.attention_backward(q, k, v, do, 0.3, True)
    a = A.attention_backward(q, k, v, do, 0.3, True, rows=np.arange(0, 13))
    b = A.attention_backward(q, k, v, do, 0.3, True, rows=np.arange(13, 40), row_block=5)
    np.testing.assert_allclose(a[1] + b[1], full[1], atol=1e-13)
    np.testing.assert_allclose(a[2] + b[2], full[2], atol=1e-13)
    np.testing.assert_allclose(a[0][:, :13], full[0][:, :13], atol=1e-14)
    np.testing.assert_allclose(b[0][:, 13:], full[0][:, 13:], atol=1e-14)
    assert np.isnan(a[0][:, 13:]).all()
