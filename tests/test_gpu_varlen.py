"""GPU parity of packed variable-length attention (forward and backward) against
the fp64 oracle, through fa_fwd_varlen / fa_bwd_varlen.

Covers length mixes with ragged tiles, one-token and empty sequences, causal
(equal lengths) and non-causal with different query and key lengths
(including keys with no queries: zero gradients), grouped heads, d = 64 and
128, the residual, a long-tailed mix at larger size on sampled sequences, and
lengths the arrays cannot hold (reported through the workspace status).
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.library().fa_set_wait_timeout_ns(10_000_000_000)


def packed_inputs(lens_q, lens_k, Hq, Hkv, d, seed):
    """Seeded bf16 tensors [total, H, d] (the inputs recipe on a batch of one)."""
    tq, tk = sum(lens_q), sum(lens_k)
    x = inputs.shape_inputs(1, Hq, Hkv, max(tq, 1), max(tk, 1), d, seed=seed)
    q, do = x["q"][0, :tq], x["do"][0, :tq]
    k, v = x["k"][0, :tk], x["v"][0, :tk]
    cq = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    ck = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return q, k, v, do, cq, ck


def run(q, k, v, do, cq, ck, max_q, max_k, causal, scale):
    dev = [t.to(DEV).contiguous() for t in (q, k, v, do, cq, ck)]
    qd, kd, vd, dod, cqd, ckd = dev
    o, lse, res = fa.forward_varlen(qd, kd, vd, cqd, ckd, max_q, max_k, causal=causal, scale=scale, residual=True)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, cqd, ckd, max_q, max_k, o, lse, dod, causal=causal, scale=scale,
                                    o_residual=res)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


CASES = [  # lens_q, lens_k, Hq, Hkv, d, causal
    ([5, 300, 128, 1, 257, 0, 129], None, 2, 2, 64, True),
    ([200, 17, 384], None, 4, 2, 128, True),
    ([100, 256, 3], [257, 40, 129], 2, 1, 128, False),
    ([130, 0, 64], [70, 200, 1], 4, 4, 64, False),      # the middle sequence has keys but no queries
    ([1000], None, 8, 2, 128, True),
]


@pytest.mark.parametrize("lens_q,lens_k,Hq,Hkv,d,causal", CASES)
def test_varlen_forward_backward(lens_q, lens_k, Hq, Hkv, d, causal):
    lens_k = lens_q if lens_k is None else lens_k
    q, k, v, do, cq, ck = packed_inputs(lens_q, lens_k, Hq, Hkv, d, seed=sum(lens_q) + d)
    scale = 1 / np.sqrt(d)
    o, lse, dq, dk, dv = run(q, k, v, do, cq, ck, max(lens_q), max(lens_k), causal, scale)
    o_ref, lse_ref = A.attention_varlen_forward(q, k, v, cq.numpy(), ck.numpy(), scale, causal)
    tag = f"varlen q={lens_q} k={lens_k} {Hq}/{Hkv} d={d} causal={causal}"
    live = np.concatenate([np.arange(cq[b], cq[b + 1]) for b in range(len(lens_q)) if lens_k[b] > 0])
    assert_fwd(o[live], lse[:, live], o_ref[live], lse_ref[:, live], tag)
    rq, rk, rv = A.attention_varlen_backward(q, k, v, do, cq.numpy(), ck.numpy(), scale, causal)
    assert_grad(dq[live], rq[live], "dQ " + tag)
    assert_grad(dk, rk, "dK " + tag)
    assert_grad(dv, rv, "dV " + tag)
    for b in range(len(lens_q)):                                 # keys no query sees: exactly zero
        if lens_q[b] == 0 and lens_k[b] > 0:
            assert not dk[ck[b]:ck[b + 1]].any() and not dv[ck[b]:ck[b + 1]].any()


def test_one_sequence_equals_dense():
    N, d = 384, 128
    q, k, v, do, cq, ck = packed_inputs([N], [N], 4, 2, d, seed=9)
    o, lse, dq, dk, dv = run(q, k, v, do, cq, ck, N, N, True, 0.1)
    qd, kd, vd, dod = (t.to(DEV)[None] for t in (q, k, v, do))
    o2, lse2, res2 = fa.forward(qd, kd, vd, causal=True, scale=0.1, residual=True)
    g2 = fa.backward(qd, kd, vd, o2, lse2, dod, causal=True, scale=0.1, o_residual=res2)
    torch.cuda.synchronize()
    assert torch.equal(o, o2[0]) and torch.equal(lse, lse2[0])
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b[0])


@pytest.mark.slow
def test_long_tailed_mix_sampled():
    """A long-tailed length mix (SFT-like, §18.7.1) at larger size; the oracle checks a few sequences."""
    g = np.random.default_rng(4)
    lens = np.clip((g.pareto(1.2, 24) + 1) * 256, 16, 4096).astype(int).tolist()
    Hq, Hkv, d = 8, 2, 128
    q, k, v, do, cq, ck = packed_inputs(lens, lens, Hq, Hkv, d, seed=4)
    scale = 1 / np.sqrt(d)
    o, lse, dq, dk, dv = run(q, k, v, do, cq, ck, max(lens), max(lens), True, scale)
    for b in (int(np.argmax(lens)), int(np.argmin(lens)), 5):
        sl_q = slice(int(cq[b]), int(cq[b + 1]))
        o_ref, lse_ref = A.attention_forward(q[None, sl_q], k[None, sl_q], v[None, sl_q], scale, True)
        assert_fwd(o[sl_q], lse[:, sl_q], o_ref[0], lse_ref[0], f"seq {b} len {lens[b]}")
        rq, rk, rv = A.attention_backward(q[None, sl_q], k[None, sl_q], v[None, sl_q], do[None, sl_q], scale, True)
        assert_grad(dq[sl_q], rq[0], f"dQ seq {b}")
        assert_grad(dk[sl_q], rk[0], f"dK seq {b}")
        assert_grad(dv[sl_q], rv[0], f"dV seq {b}")


@pytest.mark.parametrize("bad", ["longer_than_max", "causal_unequal", "past_total"])
def test_lengths_the_arrays_cannot_hold_are_reported(bad):
    lens = [100, 200]
    q, k, v, do, cq, ck = packed_inputs(lens, lens, 2, 2, 64, seed=1)
    max_q = max_k = 200
    causal = False
    if bad == "longer_than_max":
        max_q = max_k = 150
    elif bad == "causal_unequal":
        causal = True
        ck = torch.tensor([0, 120, 300], dtype=torch.int32)
    else:
        cq = torch.tensor([0, 100, 400], dtype=torch.int32)
    qd, kd, vd, cqd, ckd = (t.to(DEV).contiguous() for t in (q, k, v, cq, ck))
    s = fa.binding._varlen_shape(qd, kd, cqd, None, causal)
    o = torch.zeros_like(qd)
    lse = torch.zeros((2, qd.shape[0]), dtype=torch.float32, device=DEV)
    ws = torch.zeros(fa.library().fa_fwd_varlen_workspace_size(fa.binding.ctypes.byref(s), max_q), dtype=torch.uint8,
                     device=DEV)
    fa.fa_fwd_varlen(qd, kd, vd, cqd, ckd, max_q, max_k, o, lse, s, ws)
    rc, st = fa.binding.device_status(ws)
    assert rc == 1 and st == 0x100                             # FA_ERR_INVALID, input error only
