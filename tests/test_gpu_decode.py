"""GPU parity of split-KV decode against the fp64 oracle (through the C ABI).

Checks the final output, the per-split partials (against the oracle's
FlashDecoding statistics for the same split plan), the split boundaries
bit-exactly, and the full decode workloads on sampled heads.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from exact_io_aware_21_gb300.binding import shape
from oracle import attention as A
from oracle import plan as P
from parity import assert_fwd, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def partials(ws, s, S):
    lo, oo = ctypes.c_size_t(), ctypes.c_size_t()
    fa.binding.check(fa.library().fa_decode_partials_layout(ctypes.byref(s), S, ctypes.byref(lo), ctypes.byref(oo)))
    n = s.B * s.Hq * s.Nq * S
    lse = ws[lo.value:lo.value + 4 * n].view(torch.float32).reshape(s.B, s.Hq, s.Nq, S)
    o = ws[oo.value:oo.value + 4 * n * s.d].view(torch.float32).reshape(s.B, s.Hq, s.Nq, S, s.d)
    return lse, o


def run_decode(q, k, v, S):
    s = fa.binding._dims(q, k, None, False)
    n_used = fa.library().fa_decode_num_splits(ctypes.byref(s), S)
    ws = torch.zeros(fa.library().fa_decode_workspace_size(ctypes.byref(s), S), dtype=torch.uint8, device=DEV)
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((s.B, s.Hq, s.Nq), float("nan"), dtype=torch.float32, device=DEV)
    fa.binding.fa_decode(q, k, v, o, lse, s, S, ws)
    rc, st = fa.binding.device_status(ws)
    assert rc == 0 and st == 0
    return o, lse, ws, s, n_used


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, splits
    (1, 4, 1, 1, 1000, 128, 3),
    (2, 8, 2, 4, 1000, 128, 5),    # 16 packed rows
    (1, 2, 2, 1, 129, 64, 2),
    (2, 4, 4, 2, 5000, 64, 7),
    (1, 16, 1, 1, 300, 128, 1),    # 16 heads on one K/V head
    (1, 4, 1, 3, 4096, 128, 0),    # automatic split count
    (1, 1, 1, 1, 1, 128, 1),
    # more than 16 packed rows: two or four 16-row tiles per CTA
    (2, 8, 1, 4, 3000, 128, 4),    # 32 rows
    (1, 16, 2, 4, 1500, 128, 0),   # 32 rows, automatic splits
    (2, 16, 1, 4, 2000, 128, 3),   # 64 rows
    (1, 8, 1, 5, 777, 64, 2),      # 40 rows (a partly empty fourth tile), d = 64
    (1, 4, 4, 9, 300, 64, 1),      # 36 rows of 4 heads x 9 positions, ragged keys
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,S", CASES)
def test_decode_small(B, Hq, Hkv, Nq, Nk, d, S):
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nk + S, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse, ws, s, n_used = run_decode(q, k, v, S)
    scale = 1 / np.sqrt(d)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], scale)
    assert_fwd(o, lse, o_ref, lse_ref, f"decode {B}x{Hq}/{Hkv}x{Nq}x{Nk}x{d} S={S}")
    if S > 0:
        splits = P.decode_splits(Nk, S)
        assert len(splits) == n_used
        m, l, Ot = A.decode_partials(x["q"], x["k"], x["v"], scale, splits)
        lse_p, o_p = partials(ws, s, n_used)
        np.testing.assert_allclose(f64(lse_p), m + np.log(l), atol=1e-3, rtol=0)
        ref = Ot / l[..., None]
        err = np.linalg.norm(f64(o_p) - ref) / np.linalg.norm(ref)
        assert err < 5e-3


@pytest.mark.parametrize("Nk,S", [(1000, 3), (131072, 19), (700, 4)])
def test_split_boundaries_bit_exact(Nk, S):
    """Q = 0: each split's partial LSE is ln(its key count), so its exp is the split length."""
    B, Hq, Hkv, d = 1, 4, 1, 128
    q = torch.zeros(B, 1, Hq, d, dtype=torch.bfloat16, device=DEV)
    k = torch.randn(B, Nk, Hkv, d, device=DEV).to(torch.bfloat16)
    v = torch.randn(B, Nk, Hkv, d, device=DEV).to(torch.bfloat16)
    _, lse, ws, s, n_used = run_decode(q, k, v, S)
    lse_p, _ = partials(ws, s, n_used)
    lengths = [e - b for b, e in P.decode_splits(Nk, S)]
    got = np.rint(np.exp(f64(lse_p))).astype(np.int64)
    assert np.array_equal(got, np.broadcast_to(np.array(lengths), got.shape))
    assert np.array_equal(np.rint(np.exp(f64(lse))).astype(np.int64), np.full((B, Hq, 1), Nk))


def test_more_than_64_packed_rows_is_rejected():
    s = fa.binding.shape(1, 16, 1, 5, 1000, 128)   # 80 packed rows
    q = torch.zeros(1, 5, 16, 128, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(1, 1000, 1, 128, dtype=torch.bfloat16, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty(1, 16, 5, dtype=torch.float32, device=DEV)
    ws = torch.zeros(fa.library().fa_decode_workspace_size(ctypes.byref(s), 2), dtype=torch.uint8, device=DEV)
    with pytest.raises(fa.binding.FAError) as e:
        fa.binding.fa_decode(q, kv, kv, o, lse, s, 2, ws)
    assert e.value.code == 1


@pytest.mark.slow
def test_speculative_decode_64_rows_sampled():
    """Grouped heads x query positions = 64 packed rows (8 heads per K/V head, 8 positions)
    against a long cache: four 16-row tiles per CTA."""
    w = inputs.Workload("spec", 2, 32, 4, 8, 65536, 128, False, decode=True, seed=5)
    x = inputs.make(w, device=DEV, with_do=False)
    o, lse, _, _, _ = run_decode(x["q"], x["k"], x["v"], 0)
    for b, kvh in [(0, 0), (1, 3)]:
        hs = slice(kvh * 8, (kvh + 1) * 8)
        o_ref, lse_ref = A.attention_forward(x["q"][b:b + 1, :, hs].cpu(), x["k"][b:b + 1, :, kvh:kvh + 1].cpu(),
                                             x["v"][b:b + 1, :, kvh:kvh + 1].cpu(), w.scale)
        assert_fwd(o[b:b + 1, :, hs], lse[b:b + 1, hs], o_ref, lse_ref, f"64 rows b{b} kvh{kvh}")


@pytest.mark.slow
@pytest.mark.parametrize("w", [inputs.DECODE_Q1, inputs.DECODE_Q4], ids=lambda w: w.name)
def test_full_decode_sampled(w):
    x = inputs.make(w, device=DEV, with_do=False)
    q, k, v = x["q"], x["k"], x["v"]
    o, lse, _, _, _ = run_decode(q, k, v, 0)
    rng = np.random.default_rng(3)
    for b, kvh in [(0, 0), (int(rng.integers(w.B)), int(rng.integers(w.Hkv))), (w.B - 1, w.Hkv - 1)]:
        g = w.Hq // w.Hkv
        hs = slice(kvh * g, (kvh + 1) * g)
        qs, ks, vs = q[b:b + 1, :, hs].cpu(), k[b:b + 1, :, kvh:kvh + 1].cpu(), v[b:b + 1, :, kvh:kvh + 1].cpu()
        o_ref, lse_ref = A.attention_forward(qs, ks, vs, w.scale)
        assert_fwd(o[b:b + 1, :, hs], lse[b:b + 1, hs], o_ref, lse_ref, f"{w.name} b{b} kvh{kvh}")
    assert torch.isfinite(o).all()
