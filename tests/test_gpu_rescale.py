"""GPU parity of conditional rescaling (fa_shape_t.rescale_threshold > 0) against
the fp64 oracle: the L21 notes' FA4 variant of the online softmax, which skips
most rescalings of O by letting the exponent's reference lag the running max by
up to the threshold.

In exact arithmetic the result does not depend on the reference (the oracle's
conditional loop is pinned to the plain definition), so the forward must meet
the same bar as the exact-max forward: O rel-Frobenius <= 5e-3, max-abs <= 1e-2
beyond bf16 rounding, LSE max-abs <= 1e-3.  Covered: the tiny workload, ragged
dense shapes (d = 64 and 128, causal or not, grouped heads, Nq != Nk), a sliding
window, packed sequences, a block-sparse table, the FP8 forward (P's scale then
2^threshold / 448) against exact attention, the causal N = 4096 workload on
sampled rows, and the backward run from a thresholded forward on N(0,1) inputs
(dQ, dK, dV rel-Frobenius <= 2e-2).  On inputs whose rows are nearly one-hot
(the outlier workload) the backward from a thresholded forward is not held to
that bar: the dominant P is no longer exactly 1.0, and D = dO . O inherits its
rounding (measured envelope in the design notes); the forward still is.
"""

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd, assert_grad, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TAU = 8.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.library().fa_set_wait_timeout_ns(10_000_000_000)


DENSE = [  # B, Hq, Hkv, Nq, Nk, d, causal, tau
    (1, 1, 1, 256, 256, 64, False, TAU),      # the tiny workload's shape
    (2, 4, 2, 700, 700, 128, True, TAU),
    (1, 4, 4, 300, 300, 64, False, TAU),
    (1, 2, 2, 200, 700, 128, False, TAU),
    (1, 8, 2, 1024, 1024, 128, True, 16.0),
    (2, 2, 1, 513, 513, 64, True, 1.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,tau", DENSE)
def test_forward_and_backward_match_oracle(B, Hq, Hkv, Nq, Nk, d, causal, tau):
    x = inputs.make(inputs.TINY) if (B, Hq, Nq, d) == (1, 1, 256, 64) else \
        inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq + Hq + d)
    scale = 1 / np.sqrt(d)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse, res = fa.forward(q, k, v, causal=causal, scale=scale, residual=True, rescale_threshold=tau)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, o_residual=res)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], scale, causal)
    tag = f"{B}x{Hq}/{Hkv}x{Nq}x{Nk} d{d} causal={causal} tau={tau}"
    assert_fwd(o, lse, o_ref, lse_ref, tag, o_res=res)
    dq_ref, dk_ref, dv_ref = A.attention_backward(x["q"], x["k"], x["v"], x["do"], scale, causal)
    for g, r, n in ((dq, dq_ref, "dQ"), (dk, dk_ref, "dK"), (dv, dv_ref, "dV")):
        assert_grad(g, r, f"{n} {tag}")


def test_threshold_zero_is_the_exact_kernel():
    """A zero threshold is the default path: bit for bit the same output."""
    x = inputs.shape_inputs(1, 4, 2, 900, 900, 128, seed=77, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    a = fa.forward(q, k, v, causal=True)
    b = fa.forward(q, k, v, causal=True, rescale_threshold=0.0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_sliding_window():
    x = inputs.shape_inputs(1, 4, 2, 1000, 1000, 128, seed=5, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=True, window=(300, 0), rescale_threshold=TAU)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], 1 / np.sqrt(128), True, window=(300, 0))
    assert_fwd(o, lse, o_ref, lse_ref, "window")


def test_packed_sequences():
    lens = [200, 17, 384, 1]
    x = inputs.shape_inputs(1, 4, 2, sum(lens), sum(lens), 128, seed=6, with_do=False)
    q, k, v = (x[n][0].to(DEV).contiguous() for n in ("q", "k", "v"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    o, lse = fa.forward_varlen(q, k, v, cu, cu, max(lens), max(lens), causal=True, rescale_threshold=TAU)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_varlen_forward(x["q"][0], x["k"][0], x["v"][0], cu.cpu().numpy(),
                                                cu.cpu().numpy(), 1 / np.sqrt(128), True)
    assert_fwd(o, lse, o_ref, lse_ref, "varlen")


def test_block_sparse():
    g = np.random.default_rng(3)
    N = 1000
    nt = -(-N // 128)
    M = g.random((nt, nt)) < 0.5
    M[np.arange(nt), np.arange(nt)] = True
    rows = [np.flatnonzero(r) for r in M]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.concatenate(rows).astype(np.int32)
    x = inputs.shape_inputs(1, 4, 2, N, N, 128, seed=8, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.forward_blocksparse(q, k, v, torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV),
                                    causal=True, rescale_threshold=TAU)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_blocksparse_forward(x["q"], x["k"], x["v"], rp, ci, 1 / np.sqrt(128), True)
    assert_fwd(o, lse, o_ref, lse_ref, "block-sparse")


@pytest.mark.parametrize("had", [False, True])
def test_fp8_forward(had):
    """E4M3 operands: P enters P V as E4M3(448 P / 2^threshold).  Held to the FP8 scheme's
    own bound against exact attention, and to the pages' Table 18-21 level (MSE < 5e-5)."""
    w = inputs.Workload("t", 1, 8, 2, 1024, 1024, 128, True, seed=9)
    x = inputs.make(w, with_do=False)
    sg = inputs.hadamard_signs(128, seed=128).to(DEV) if had else None
    q8, sq = fa.quantize_fp8(x["q"].to(DEV), 128, sg)
    k8, sk = fa.quantize_fp8(x["k"].to(DEV), 128, sg)
    v8, sv = fa.quantize_fp8(x["v"].to(DEV), 0, None)
    scale = 1 / np.sqrt(128)
    o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=scale, rescale_threshold=TAU)
    o0, lse0 = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=scale)
    torch.cuda.synchronize()
    o_ex, lse_ex = A.attention_forward(x["q"], x["k"], x["v"], scale, True)
    o_f, o0_f = o.float().cpu().numpy(), o0.float().cpu().numpy()
    assert np.isfinite(o_f).all() and np.isfinite(lse.cpu().numpy()).all()
    assert rel_fro(o, o_ex) < 0.08
    mse, mse0 = float(np.mean((o_f - o_ex) ** 2)), float(np.mean((o0_f - o_ex) ** 2))
    assert mse < 5e-5 and mse < 2.0 * mse0, (mse, mse0)
    # LSE: within the FP8 scheme's own error at the exact running max (E4M3 scores)
    e_lse = float(np.abs(lse.cpu().numpy() - lse_ex).max())
    e_lse0 = float(np.abs(lse0.cpu().numpy() - lse_ex).max())
    assert e_lse <= 1.25 * e_lse0 + 1e-3, (e_lse, e_lse0)


@pytest.mark.slow
def test_causal_n4096_sampled():
    w = inputs.CAUSAL_N4096_D128
    x = inputs.make(w, device=DEV, with_do=False)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, scale=w.scale, rescale_threshold=TAU)
    torch.cuda.synchronize()
    heads = [(0, 0), (1, 15)]
    rows = np.concatenate([np.arange(0, 128), np.arange(2048, 2176), np.arange(3968, 4096)])
    o_ref, lse_ref = A.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), w.scale, True, heads=heads,
                                         rows=rows)
    for b, h in heads:
        assert_fwd(o[b, rows, h], lse[b, h, rows], o_ref[b, rows, h], lse_ref[b, h, rows], f"N4096 b{b} h{h}")


def test_outlier_rows_forward_meets_the_bar():
    """Nearly one-hot rows (outlier channel x20 in Q and K): the thresholded forward still
    meets the forward bar (its backward is outside the 2e-2 envelope; see the module note)."""
    w = inputs.Workload("o", 1, 4, 1, 2048, 2048, 128, True, outliers=True, seed=0)
    x = inputs.make(w, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse, res = fa.forward(q, k, v, causal=True, residual=True, rescale_threshold=TAU)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], w.scale, True)
    assert_fwd(o, lse, o_ref, lse_ref, "outliers", o_res=res)
