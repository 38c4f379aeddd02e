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


def assert_fwd(o, lse, o_ref, lse_ref, what=""):
    o, lse, o_ref, lse_ref = f64(o), f64(lse), f64(o_ref), f64(lse_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{what}: non-finite output"
    e1, e2, e3 = rel_fro(o, o_ref), max_abs(o, o_ref), max_abs(lse, lse_ref)
    assert e1 <= O_REL_FRO and e2 <= O_MAX_ABS and e3 <= LSE_MAX_ABS, \
        f"{what}: O rel-fro {e1:.2e} (<= {O_REL_FRO}), O max-abs {e2:.2e} (<= {O_MAX_ABS}), " \
        f"LSE max-abs {e3:.2e} (<= {LSE_MAX_ABS})"


def assert_grad(g, ref, what=""):
    g, ref = f64(g), f64(ref)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    e = rel_fro(g, ref)
    assert e <= GRAD_REL_FRO, f"{what}: rel-fro {e:.2e} (<= {GRAD_REL_FRO})"
