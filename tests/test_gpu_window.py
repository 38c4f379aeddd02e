"""GPU parity of sliding-window attention (forward and backward) against the fp64 oracle.

Windows narrower than a tile, wider than the sequence, one-sided, zero-width,
with and without causal, on ragged lengths and grouped heads; the exact key
count per row recovered from LSE with Q = 0; and a long causal sliding window
on sampled rows.
"""

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd, assert_grad

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # B, Hq, Hkv, N, d, window, causal
    (1, 2, 2, 1000, 64, (100, 50), False),
    (2, 4, 2, 777, 128, (300, -1), True),
    (1, 4, 4, 512, 64, (0, 0), False),
    (1, 8, 2, 2048, 128, (256, 256), False),
    (1, 2, 1, 300, 128, (1000, 3), True),
    (1, 4, 4, 1500, 128, (384, 0), True),
    (1, 2, 2, 640, 64, (128, -1), False),
    (2, 2, 1, 1029, 128, (-1, 200), False),
    (1, 1, 1, 129, 64, (5, 5), False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,window,causal", CASES)
def test_window_forward_backward(B, Hq, Hkv, N, d, window, causal):
    x = inputs.shape_inputs(B, Hq, Hkv, N, N, d, seed=N + d + window[0])
    scale = 1 / np.sqrt(d)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse, res = fa.forward(q, k, v, causal=causal, scale=scale, residual=True, window=window)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, o_residual=res, window=window)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], scale, causal, window=window)
    tag = f"{B}x{Hq}/{Hkv}x{N}x{d} window={window} causal={causal}"
    assert_fwd(o, lse, o_ref, lse_ref, tag)
    rq, rk, rv = A.attention_backward(x["q"], x["k"], x["v"], x["do"], scale, causal, window=window)
    for g, ref, name in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        if np.linalg.norm(ref) == 0:  # a one-key window: P = 1, dS = 0, so dQ = dK = 0 exactly
            assert float(g.abs().max()) <= 1e-5, f"{name} {tag}: {float(g.abs().max()):.2e} (exact 0)"
        else:
            assert_grad(g, ref, f"{name} {tag}")


@pytest.mark.parametrize("window,causal", [((100, 50), False), ((300, 0), True), ((0, 0), False),
                                           ((129, 255), False)])
def test_zero_query_counts_window_keys_exactly(window, causal):
    N, d = 1000, 64
    x = inputs.shape_inputs(1, 2, 2, N, N, d, seed=4, with_do=False)
    q = torch.zeros(1, N, 2, d, dtype=torch.bfloat16, device=DEV)
    _, lse = fa.forward(q, x["k"].to(DEV), x["v"].to(DEV), causal=causal, scale=1.0, window=window)
    i = np.arange(N)
    lo = np.maximum(0, i - window[0]) if window[0] >= 0 else np.zeros(N, dtype=int)
    hi = np.minimum(N - 1, i + window[1]) if window[1] >= 0 else np.full(N, N - 1)
    if causal:
        hi = np.minimum(hi, i)
    counts = torch.round(torch.exp(lse.double())).long().cpu().numpy()
    assert (counts == (hi - lo + 1)[None, None, :]).all()


@pytest.mark.slow
def test_long_causal_sliding_window_sampled():
    B, Hq, Hkv, N, d, window = 1, 8, 2, 8192, 128, (2048, 0)
    x = inputs.shape_inputs(B, Hq, Hkv, N, N, d, seed=99, device=DEV)
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    scale = 1 / np.sqrt(d)
    o, lse, res = fa.forward(q, k, v, causal=True, scale=scale, residual=True, window=window)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, o_residual=res, window=window)
    torch.cuda.synchronize()
    qc, kc, vc, doc = q.cpu(), k.cpu(), v.cpu(), do.cpu()
    rows = np.array([0, 1, 127, 2047, 2048, 2049, 5000, N - 1])
    keys = np.array([0, 2047, 5000, N - 1])
    g = Hq // Hkv
    kv = 1
    dk_ref = np.zeros((len(keys), d))
    dv_ref = np.zeros((len(keys), d))
    for h in range(kv * g, (kv + 1) * g):
        o_ref, lse_ref = A.attention_forward(qc, kc, vc, scale, True, heads=[(0, h)], rows=rows, window=window)
        assert_fwd(o[0, rows, h], lse[0, h, rows], o_ref[0, rows, h], lse_ref[0, h, rows], f"long window O h{h}")
        rq, rk, rv = A.attention_backward_sampled(qc, kc, vc, doc, scale, True, 0, h, rows, keys, window=window)
        assert_grad(dq[0, rows, h], rq, f"long window dQ h{h}")
        dk_ref += rk
        dv_ref += rv
    assert_grad(dk[0, keys, kv], dk_ref, "long window dK")
    assert_grad(dv[0, keys, kv], dv_ref, "long window dV")
