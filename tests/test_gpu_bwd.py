"""GPU parity of the backward kernels against the fp64 oracle (through the C ABI).

The GPU backward consumes the GPU forward's O and LSE (as a caller would); the
oracle recomputes everything from Q, K, V, dO in fp64.
"""

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_grad, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(x, causal, scale, residual=True):
    """Forward then backward on the GPU; with the residual unless told otherwise."""
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse, res = fa.forward(q, k, v, causal=causal, scale=scale, residual=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, o_residual=res if residual else None)
    torch.cuda.synchronize()
    return dq, dk, dv


def test_tiny_workload():
    w = inputs.TINY
    x = inputs.make(w)
    dq, dk, dv = run(x, w.causal, w.scale)
    rq, rk, rv = A.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
    assert_grad(dq, rq, "dQ")
    assert_grad(dk, rk, "dK")
    assert_grad(dv, rv, "dV")


CASES = [
    # B, Hq, Hkv, N(q=k), d, causal
    (1, 1, 1, 128, 64, False),
    (1, 2, 2, 256, 128, True),
    (2, 3, 3, 300, 64, True),
    (1, 4, 2, 1000, 128, True),
    (2, 2, 1, 513, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 1, 1, 127, 64, False),
    (1, 8, 1, 384, 128, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", CASES)
def test_small_shapes(B, Hq, Hkv, N, d, causal):
    x = inputs.shape_inputs(B, Hq, Hkv, N, N, d, seed=N + d + Hq)
    scale = 1 / np.sqrt(d)
    dq, dk, dv = run(x, causal, scale)
    rq, rk, rv = A.attention_backward(x["q"], x["k"], x["v"], x["do"], scale, causal)
    tag = f"{B}x{Hq}/{Hkv}x{N}x{d} causal={causal}"
    assert_grad(dq, rq, "dQ " + tag)
    assert_grad(dk, rk, "dK " + tag)
    assert_grad(dv, rv, "dV " + tag)


@pytest.mark.parametrize("causal", [False, True])
def test_without_residual(causal):
    """Without O's residual D comes from bf16 O; on N(0,1) inputs that is still in bounds."""
    x = inputs.shape_inputs(1, 4, 2, 600, 600, 128, seed=31)
    dq, dk, dv = run(x, causal, 0.088, residual=False)
    rq, rk, rv = A.attention_backward(x["q"], x["k"], x["v"], x["do"], 0.088, causal)
    assert_grad(dq, rq, "dQ")
    assert_grad(dk, rk, "dK")
    assert_grad(dv, rv, "dV")


def test_bwd_parts_equal_bwd():
    """fa_bwd_part 0, 1, 2 in order gives bit-identical gradients to fa_bwd."""
    import ctypes

    x = inputs.shape_inputs(1, 4, 2, 700, 700, 64, seed=8)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse, res = fa.forward(q, k, v, causal=True, residual=True)
    a = fa.backward(q, k, v, o, lse, do, causal=True, o_residual=res)
    s = fa.binding._dims(q, k, None, True)
    ws = torch.zeros(fa.library().fa_bwd_workspace_size(ctypes.byref(s)), dtype=torch.uint8, device=DEV)
    g = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    for part in range(3):
        fa.binding.fa_bwd_part(part, q, k, v, o, lse, do, *g, s, ws, res)
    torch.cuda.synchronize()
    for u, w in zip(a, g):
        assert torch.equal(u, w)


def test_rectangular_noncausal():
    x = inputs.shape_inputs(1, 2, 2, 200, 700, 128, seed=9)
    dq, dk, dv = run(x, False, 0.088)
    rq, rk, rv = A.attention_backward(x["q"], x["k"], x["v"], x["do"], 0.088, False)
    assert_grad(dq, rq, "dQ")
    assert_grad(dk, rk, "dK")
    assert_grad(dv, rv, "dV")


def test_zero_upstream_gives_zero_gradients():
    x = inputs.shape_inputs(1, 2, 1, 300, 300, 128, seed=2)
    x["do"] = torch.zeros_like(x["do"])
    dq, dk, dv = run(x, True, 0.1)
    assert not dq.any() and not dk.any() and not dv.any()


def test_deterministic():
    x = inputs.shape_inputs(1, 4, 2, 700, 700, 128, seed=4)
    a = run(x, True, 0.1)
    b = run(x, True, 0.1)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.slow
@pytest.mark.parametrize("w", [inputs.MHA_N2048_D64, inputs.CAUSAL_N4096_D128, inputs.GQA_N8192_D128],
                         ids=lambda w: w.name)
def test_full_workload_sampled(w):
    """Full-size backward; sampled rows of dQ and of one K/V head's dK, dV."""
    x = inputs.make(w)
    dq, dk, dv = run(x, w.causal, w.scale)
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    rng = np.random.default_rng(17)
    g = w.Hq // w.Hkv
    b, kvh = int(rng.integers(w.B)), int(rng.integers(w.Hkv))
    q_rows = np.unique(np.concatenate([[0, w.Nq - 1], rng.integers(0, w.Nq, 48)]))
    k_rows = np.unique(np.concatenate([[0, w.Nk - 1], rng.integers(0, w.Nk, 48)]))
    sk = np.zeros((len(k_rows), w.d))
    sv = np.zeros((len(k_rows), w.d))
    for h in range(kvh * g, (kvh + 1) * g):
        rq, rk, rv = A.attention_backward_sampled(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal, b, h,
                                                  q_rows, k_rows)
        assert_grad(dq[b, q_rows, h], rq, f"dQ b{b} h{h}")
        sk += rk
        sv += rv
    assert_grad(dk[b, k_rows, kvh], sk, f"dK b{b} kvh{kvh}")
    assert_grad(dv[b, k_rows, kvh], sv, f"dV b{b} kvh{kvh}")
