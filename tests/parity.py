"""Parity metrics and tolerances shared by the GPU tests.

Tolerances (the acceptance bar for bf16 inputs against the fp64 oracle):
forward O relative Frobenius error <= 5e-3 and max abs error <= 1e-2; LSE max
abs error <= 1e-3; dQ, dK, dV relative Frobenius error <= 2e-2.  Integer work
(masks, split boundaries) must match exactly.
"""

import numpy as np
import torch

O_REL_FRO = 5e-3
O_MAX_ABS = 1e-2
LSE_MAX_ABS = 1e-3
GRAD_REL_FRO = 2e-2


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def rel_fro(x, ref):
    x, ref = f64(x), f64(ref)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(x, ref):
    return float(np.abs(f64(x) - f64(ref)).max())


def half_ulp_bf16(x):
    """Half a bf16 unit in the last place at |x| (8 significant bits)."""
    a = np.abs(f64(x))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def assert_fwd(o, lse, o_ref, lse_ref, what="", o_res=None):
    """Forward bar.  O is a bf16 output, so its max-abs bound is read as 1e-2
    beyond bf16's own rounding of the exact value (half an ulp at |O_ref|, which
    alone exceeds 1e-2 once |O| >= 4).  With the residual, O + residual must be
    within 1e-2 of the oracle outright."""
    o, lse, o_ref, lse_ref = f64(o), f64(lse), f64(o_ref), f64(lse_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    e1, e3 = rel_fro(o, o_ref), max_abs(lse, lse_ref)
    e2 = float(np.max(np.abs(o - o_ref) - half_ulp_bf16(o_ref)))
    assert e1 <= O_REL_FRO and e2 <= O_MAX_ABS and e3 <= LSE_MAX_ABS, \
        f"{what}: O rel-fro {e1:.2e} (<= {O_REL_FRO}), O max-abs beyond bf16 rounding {e2:.2e} " \
        f"(<= {O_MAX_ABS}), LSE max-abs {e3:.2e} (<= {LSE_MAX_ABS})"
    if o_res is not None:
        e4 = max_abs(o + f64(o_res), o_ref)
        assert e4 <= O_MAX_ABS, f"{what}: O + residual max-abs {e4:.2e} (<= {O_MAX_ABS})"


def assert_grad(g, ref, what=""):
    g, ref = f64(g), f64(ref)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    e = rel_fro(g, ref)
    assert e <= GRAD_REL_FRO, f"{what}: rel-fro {e:.2e} (<= {GRAD_REL_FRO})"
