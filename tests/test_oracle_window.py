"""Pins of the oracle's sliding-window attention (no GPU).

Reductions to the already-pinned full and causal oracles, the one-key window
(closed form), Q = 0 (prefix-free mean over the window, LSE = ln of the count),
a per-row brute force written with explicit loops, central differences of the
windowed backward, and the window tile plan against a brute-force scan.
"""

import numpy as np
import pytest

from oracle import attention as A
from oracle import plan as P

RNG = np.random.default_rng(7)


def rand(*shape):
    return RNG.standard_normal(shape)


def test_unbounded_window_is_full_attention():
    q, k, v = rand(1, 40, 2, 8), rand(1, 40, 1, 8), rand(1, 40, 1, 8)
    a = A.attention_forward(q, k, v, 0.3, window=(40, 40))
    b = A.attention_forward(q, k, v, 0.3)
    c = A.attention_forward(q, k, v, 0.3, window=(-1, -1))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(c[0], b[0]) and np.array_equal(c[1], b[1])


@pytest.mark.parametrize("right", [-1, 0, 5])
def test_causal_with_unbounded_left_is_causal(right):
    q, k, v = rand(2, 33, 2, 8), rand(2, 33, 2, 8), rand(2, 33, 2, 8)
    a = A.attention_forward(q, k, v, 0.4, causal=True, window=(-1, right))
    b = A.attention_forward(q, k, v, 0.4, causal=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_zero_window_returns_own_value():
    q, k, v = rand(1, 17, 4, 8), rand(1, 17, 2, 8), rand(1, 17, 2, 8)
    O, LSE = A.attention_forward(q, k, v, 0.5, window=(0, 0))
    for h in range(4):
        assert np.allclose(O[0, :, h], v[0, :, h // 2], atol=1e-15)
        assert np.allclose(LSE[0, h], 0.5 * np.sum(q[0, :, h] * k[0, :, h // 2], axis=-1), atol=1e-13)


@pytest.mark.parametrize("left,right,causal", [(3, 2, False), (10, -1, True), (0, 7, False), (5, 0, True)])
def test_zero_query_averages_the_window(left, right, causal):
    N = 30
    _, k, v = rand(1, N, 1, 4), rand(1, N, 1, 4), rand(1, N, 1, 4)
    q = np.zeros((1, N, 1, 4))
    O, LSE = A.attention_forward(q, k, v, 1.0, causal=causal, window=(left, right))
    for i in range(N):
        lo = 0 if left < 0 else max(0, i - left)
        hi = N - 1 if right < 0 else min(N - 1, i + right)
        if causal:
            hi = min(hi, i)
        assert np.allclose(O[0, i, 0], v[0, lo:hi + 1, 0].mean(axis=0), atol=1e-14)
        assert abs(LSE[0, 0, i] - np.log(hi - lo + 1)) < 1e-14


def test_brute_force_rows():
    N, d, left, right, scale = 23, 5, 4, 2, 0.7
    q, k, v = rand(1, N, 1, d), rand(1, N, 1, d), rand(1, N, 1, d)
    O, LSE = A.attention_forward(q, k, v, scale, window=(left, right))
    for i in range(N):
        js = [j for j in range(N) if i - left <= j <= i + right]
        s = [scale * sum(q[0, i, 0, c] * k[0, j, 0, c] for c in range(d)) for j in js]
        m = max(s)
        e = [np.exp(x - m) for x in s]
        z = sum(e)
        o = [sum(e[t] * v[0, js[t], 0, c] for t in range(len(js))) / z for c in range(d)]
        assert np.allclose(O[0, i, 0], o, atol=1e-13)
        assert abs(LSE[0, 0, i] - (m + np.log(z))) < 1e-13


@pytest.mark.parametrize("window,causal", [((2, 1), False), ((3, -1), True)])
def test_windowed_backward_finite_differences(window, causal):
    B, N, Hq, Hkv, d, scale = 1, 8, 2, 1, 4, 0.6
    q, k, v, do = rand(B, N, Hq, d), rand(B, N, Hkv, d), rand(B, N, Hkv, d), rand(B, N, Hq, d)
    dq, dk, dv = A.attention_backward(q, k, v, do, scale, causal, window=window)

    def loss(q_, k_, v_):
        return float(np.sum(A.attention_forward(q_, k_, v_, scale, causal, window=window)[0] * do))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            a = {"q": q, "k": k, "v": v}
            a[name] = xp
            fp = loss(a["q"], a["k"], a["v"])
            a[name] = xm
            fm = loss(a["q"], a["k"], a["v"])
            num[idx] = (fp - fm) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(g) < 1e-7, name


@pytest.mark.parametrize("N,left,right,causal", [(1000, 100, 50, False), (777, 300, -1, True), (512, 0, 0, False),
                                                 (640, 128, 128, False), (300, 1000, 3, True)])
def test_window_tile_plan_matches_brute_force(N, left, right, causal):
    T = 128
    nt = -(-N // T)
    for qi in range(nt):
        for kj in range(nt):
            qs, qe, ks, ke = qi * T, min(N, qi * T + T), kj * T, min(N, kj * T + T)
            vis = [(left < 0 or j >= i - left) and (right < 0 or j <= i + right) and (not causal or j <= i)
                   for i in range(qs, qe) for j in range(ks, ke)]
            exp = P.SKIP if not any(vis) else (P.FULL if all(vis) else P.PARTIAL)
            assert P.window_tile_class(qs, qe, ks, ke, left, right, causal) == exp
    ranges = P.tile_ranges(N, N, T, left, right, causal)
    for qi, (lo, hi) in enumerate(ranges):
        cls = [P.window_tile_class(qi * T, min(N, qi * T + T), kj * T, min(N, kj * T + T), left, right, causal)
               for kj in range(nt)]
        assert all(c != P.SKIP for c in cls[lo:hi]) and all(c == P.SKIP for c in cls[:lo] + cls[hi:])
