"""GPU parity of the forward kernel against the fp64 oracle (through the C ABI).

Covers: the tensor-core building blocks (self-test), small shapes spanning
several tiles with ragged tails, d = 64 and 128, causal and non-causal, grouped
heads, Nq != Nk, strided views, the bit-exact causal mask, and the workloads of
the benchmark at full size on sampled rows.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd, f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.library()
    fa.library().fa_set_wait_timeout_ns(10_000_000_000)


def status_ok(ws):
    rc, st = fa.binding.device_status(ws)
    assert rc == 0 and st == 0, f"device status {st:#x}"


# ------------------------------------------------------------------ building blocks
@pytest.mark.parametrize("k", [64, 128])
def test_selftest_qk_form(k):
    g = torch.Generator().manual_seed(k)
    a = torch.randn(128, k, generator=g).to(torch.bfloat16)
    b = torch.randn(128, k, generator=g).to(torch.bfloat16)
    c = torch.zeros(128, 128, dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    da, db = a.to(DEV), b.to(DEV)   # keep the device copies alive during the call
    fa.binding.check(fa.library().fa_selftest_mma(0, k, da.data_ptr(), db.data_ptr(), c.data_ptr(),
                                                  ws.data_ptr(), None))
    torch.cuda.synchronize()
    ref = f64(a) @ f64(b).T
    np.testing.assert_allclose(f64(c), ref, rtol=1e-5, atol=1e-4)
    status_ok(ws)


@pytest.mark.parametrize("n", [64, 128])
def test_selftest_pv_form(n):
    g = torch.Generator().manual_seed(100 + n)
    a = torch.rand(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(128, n, generator=g).to(torch.bfloat16)
    c = torch.zeros(128, n, dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    da, db = a.to(DEV), b.to(DEV)
    fa.binding.check(fa.library().fa_selftest_mma(1, n, da.data_ptr(), db.data_ptr(), c.data_ptr(),
                                                  ws.data_ptr(), None))
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(c), f64(a) @ f64(b), rtol=1e-5, atol=1e-4)
    status_ok(ws)


# ------------------------------------------------------------------ small shapes
def run_fwd(x, causal, scale, residual=False):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out = fa.forward(q, k, v, causal=causal, scale=scale, residual=residual)
    torch.cuda.synchronize()
    return out


def test_tiny_workload():
    w = inputs.TINY
    x = inputs.make(w)
    o, lse = run_fwd(x, w.causal, w.scale)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], w.scale, w.causal)
    assert_fwd(o, lse, o_ref, lse_ref, w.name)


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 1, 1, 128, 128, 64, False),
    (1, 2, 2, 256, 256, 128, True),
    (2, 3, 3, 300, 300, 64, True),      # ragged: 3 query tiles, odd pair count
    (1, 4, 2, 1000, 1000, 128, True),   # grouped heads, ragged
    (2, 2, 1, 513, 513, 64, False),
    (1, 2, 2, 200, 700, 128, False),    # Nq != Nk
    (1, 2, 2, 700, 130, 64, False),
    (1, 1, 1, 1, 1, 128, True),         # one row, one key
    (1, 1, 1, 127, 127, 64, True),
    (1, 1, 1, 129, 129, 128, True),
    (1, 8, 1, 384, 384, 128, False),    # multi-query
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", CASES)
def test_small_shapes(B, Hq, Hkv, Nq, Nk, d, causal):
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq * 7 + Nk + d, with_do=False)
    scale = 1 / np.sqrt(d)
    o, lse = run_fwd(x, causal, scale)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], scale, causal)
    assert_fwd(o, lse, o_ref, lse_ref, f"{B}x{Hq}/{Hkv}x{Nq}x{Nk}x{d} causal={causal}")


def test_strided_views_and_custom_scale():
    """Q/K/V as slices of a packed [B, N, 3, H, d] buffer (head stride != d)."""
    B, N, H, d = 2, 300, 2, 128
    g = torch.Generator().manual_seed(5)
    qkv = torch.randn(B, N, 3, H, d, generator=g).to(torch.bfloat16)
    dq = qkv.to(DEV)
    q, k, v = dq[:, :, 0], dq[:, :, 1], dq[:, :, 2]
    o, lse = fa.forward(q, k, v, causal=True, scale=0.05)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_forward(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], 0.05, True)
    assert_fwd(o, lse, o_ref, lse_ref, "strided")


@pytest.mark.parametrize("N,d", [(1000, 64), (4096, 128), (300, 128)])
def test_causal_mask_bit_exact(N, d):
    """Q = 0: every visible score is 0, so exp(LSE_i) counts the visible keys: i + 1."""
    B, H = 1, 2
    q = torch.zeros(B, N, H, d, dtype=torch.bfloat16, device=DEV)
    k = torch.randn(B, N, H, d, device=DEV).to(torch.bfloat16)
    v = torch.randn(B, N, H, d, device=DEV).to(torch.bfloat16)
    _, lse = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    counts = np.rint(np.exp(f64(lse))).astype(np.int64)
    assert np.array_equal(counts, np.broadcast_to(np.arange(1, N + 1), counts.shape))
    _, lse = fa.forward(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert np.array_equal(np.rint(np.exp(f64(lse))).astype(np.int64), np.full((B, H, N), N))


@pytest.mark.parametrize("d", [64, 128])
def test_residual_output(d):
    """The optional residual is bf16(O_fp32 - O): it is O's own rounding remainder,
    O + residual meets the bound outright, and asking for it leaves O and LSE unchanged."""
    x = inputs.shape_inputs(1, 2, 1, 500, 500, d, seed=21, with_do=False)
    o1, l1 = run_fwd(x, True, 0.1)
    o, lse, res = run_fwd(x, True, 0.1, residual=True)
    assert torch.equal(o, o1) and torch.equal(lse, l1)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], 0.1, True)
    assert_fwd(o, lse, o_ref, lse_ref, "residual", o_res=res)
    # the residual is O's own rounding remainder: at most half a bf16 ulp of O
    from parity import half_ulp_bf16

    r, hi = f64(res), f64(o)
    assert np.all(np.abs(r) <= half_ulp_bf16(hi) * (1 + 2 ** -7) + 1e-30)
    assert np.abs(r).max() > 0


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", [
    (1, 2, 2, 1000, 1000, 128), (2, 2, 2, 513, 513, 64), (1, 8, 8, 2048, 2048, 128),
    (1, 8, 2, 1024, 1024, 128),   # grouped heads, 4 parts
    (1, 4, 1, 777, 777, 64),      # one K/V head, 3 parts, the last holding the ragged tile
    (1, 2, 2, 300, 1500, 64),     # Nq != Nk, 4 parts of 3 key tiles each
])
def test_key_split_units(B, Hq, Hkv, Nq, Nk, d):
    """Without a mask the units of a partial last wave run as parts along the keys,
    merged by their LSE: O (with its residual) and LSE still meet the bound, the
    part holding the ragged last key tile included, and the workspace holds the
    parts.  (The full MHA workload, split in its last wave, is checked below.)"""
    s = fa.binding.shape(B, Hq, Hkv, Nq, Nk, d, None, False)
    s0, ns = ctypes.c_int(), ctypes.c_int()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.library().fa_fwd_split_plan(ctypes.byref(s), sms, ctypes.byref(s0), ctypes.byref(ns)) == 0
    assert ns.value >= 2  # the shape does split
    assert fa.library().fa_fwd_workspace_size(ctypes.byref(s)) > 256  # room for the parts' O and LSE
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq + Nk + d, with_do=False)
    o, lse, res = run_fwd(x, False, 1 / np.sqrt(d), residual=True)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], 1 / np.sqrt(d), False)
    assert_fwd(o, lse, o_ref, lse_ref, f"key-split {B}x{Hq}/{Hkv}x{Nq}x{Nk} d={d} parts={ns.value}", o_res=res)


@pytest.mark.parametrize("causal", [True, False])
def test_deterministic(causal):
    """Bitwise the same on a second call: the causal schedule is static and, without
    a mask, this small grid runs key-split parts merged in a fixed order."""
    x = inputs.shape_inputs(1, 4, 2, 1000, 1000, 128, seed=3, with_do=False)
    a = run_fwd(x, causal, 0.1, residual=True)
    b = run_fwd(x, causal, 0.1, residual=True)
    assert all(torch.equal(u, v) for u, v in zip(a, b))


# ------------------------------------------------------------------ full-size workloads
def sampled_check(w, n_heads=3, n_rows=96, seed=11):
    x = inputs.make(w, with_do=False)
    o, lse, res = run_fwd(x, w.causal, w.scale, residual=True)
    rng = np.random.default_rng(seed)
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.Hq))) for _ in range(n_heads)]
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.Nq - 1], rng.integers(0, w.Nq, n_rows)]))
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], w.scale, w.causal, heads=heads, rows=rows)
    for b, h in heads:
        assert_fwd(o[b, rows, h], lse[b, h, rows], o_ref[b, rows, h], lse_ref[b, h, rows], f"{w.name} b{b} h{h}",
                   o_res=res[b, rows, h])
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.slow
@pytest.mark.parametrize("w", [inputs.MHA_N2048_D64, inputs.CAUSAL_N4096_D128, inputs.GQA_N8192_D128],
                         ids=lambda w: w.name)
def test_full_workload_sampled(w):
    sampled_check(w)


# ------------------------------------------------------------------ forward trace (diagnostics)
def test_forward_trace_stamps_every_unit_and_leaves_results_unchanged():
    """A traced launch writes consistent timestamps for every CTA and unit (claimed <=
    first product <= last product <= output written, inside its CTA's span) and
    computes the same output, bit for bit, as an untraced launch."""
    x = inputs.shape_inputs(2, 4, 2, 1000, 1000, 128, seed=31, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o_ref, lse_ref = fa.forward(q, k, v, causal=True)
    s = fa.binding.shape(2, 4, 2, 1000, 1000, 128, None, True)
    units = fa.library().fa_fwd_num_units(ctypes.byref(s))
    buf = torch.zeros(fa.binding.TRACE_UNIT0 + fa.binding.TRACE_UNIT_WORDS * units, dtype=torch.int64, device=DEV)
    fa.binding.set_trace(buf)
    try:
        o, lse = fa.forward(q, k, v, causal=True)
        torch.cuda.synchronize()
    finally:
        fa.binding.set_trace(None)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    t = buf.cpu().numpy()
    cta = t[:4096].reshape(1024, 4)
    grid = int((cta[:, 0] > 0).sum())
    assert grid == min(units, torch.cuda.get_device_properties(0).multi_processor_count)
    assert (cta[:grid, 1] >= cta[:grid, 0]).all() and int(cta[:grid, 3].sum()) == units
    rec = t[4096:4096 + 16 * units].reshape(units, 16)
    assert (rec[:, 0] > 0).all() and (rec[:, 1] >= rec[:, 0]).all() and (rec[:, 2] >= rec[:, 1]).all()
    assert (rec[:, 3] >= rec[:, 2]).all()
    c = rec[:, 4]
    assert ((c >= 0) & (c < grid)).all()
    assert (rec[:, 0] >= cta[c, 0]).all() and (rec[:, 3] <= cta[c, 1]).all()
