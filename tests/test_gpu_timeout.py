"""Bounded device waits on the GPU: a wait that runs out ends the kernel with an
error status the host reads, and the process stays able to run the next call.

The failure is made without faulting anything: the library's test hook
(fa_test_withhold_arrive) runs a test instantiation of the forward kernel in
which one softmax warp of the CTA that runs work unit 0 skips its first hand-off
of P (one software mbarrier arrive).  With a 1 ms wait budget a wait of that CTA gives up (the
tensor-core issuer's, or the producer's for a stage the issuer never frees),
records its timeout bit, and the CTA's roles leave: copies in flight land and
TMEM is freed.  The next, normal call must then match the fp64
oracle, which it could not if TMEM or a copy had been left behind.
"""

import ctypes
import time

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import binding as B
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd, assert_grad, f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FA_ERR_TIMEOUT = 6
FA_STATUS_TIMEOUT_LOAD = 0x1
FA_STATUS_TIMEOUT_MMA = 0x2
FA_STATUS_TIMEOUT_MASK = 0xFF


def test_withheld_handoff_runs_out_and_the_next_call_is_exact():
    lib = fa.library()
    x = inputs.shape_inputs(1, 4, 2, 1024, 1024, 128, seed=41)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    s = B.shape(1, 4, 2, 1024, 1024, 128, None, True)
    ws = torch.zeros(lib.fa_fwd_workspace_size(ctypes.byref(s)), dtype=torch.uint8, device=DEV)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 4, 1024), float("nan"), dtype=torch.float32, device=DEV)
    lib.fa_set_wait_timeout_ns(1_000_000)  # 1 ms
    try:
        lib.fa_test_withhold_arrive()
        t0 = time.time()
        B.fa_fwd(q, k, v, o, lse, s, ws)
        rc, bits = B.device_status(ws)
        elapsed = time.time() - t0
    finally:
        lib.fa_set_wait_timeout_ns(10_000_000_000)
    # whichever of that CTA's waits started first runs out first: the tensor-core
    # issuer's (for the withheld P) or the producer's (for a stage the issuer never frees)
    assert rc == FA_ERR_TIMEOUT, f"status {bits:#x}"
    assert bits & (FA_STATUS_TIMEOUT_MMA | FA_STATUS_TIMEOUT_LOAD), f"status {bits:#x}"
    assert not (bits & ~FA_STATUS_TIMEOUT_MASK), f"status {bits:#x}"
    assert elapsed < 5.0
    # that CTA gave up on its units: their rows stay unwritten (NaN); every row that was
    # written is a complete, exact row (an epilogue runs only after all its products)
    o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], s.scale, True)
    rows_nan = torch.isnan(lse).cpu().numpy()  # [B, Hq, Nq]
    assert rows_nan[0, 0, 768:].all()  # unit 0, causal: query tiles 6 and 7 of head 0 (longest first)
    done = ~rows_nan[0].T  # [Nq, Hq]
    assert_fwd(f64(o)[0][done], f64(lse)[0].T[done], o_ref[0][done], lse_ref[0].T[done], "rows written")

    # the hook is one-shot: the next calls run the normal kernels, exactly
    ws2 = torch.zeros_like(ws)
    o2 = torch.full_like(q, float("nan"))
    lse2 = torch.full_like(lse, float("nan"))
    B.fa_fwd(q, k, v, o2, lse2, s, ws2)
    assert B.device_status(ws2) == (0, 0)
    assert_fwd(o2, lse2, o_ref, lse_ref, "forward after the timeout")
    # the workspace that recorded the timeout: the next call clears its header first
    # (a kernel the forward's set-up overlaps), so the status is that call's own
    o4 = torch.full_like(q, float("nan"))
    lse4 = torch.full_like(lse, float("nan"))
    B.fa_fwd(q, k, v, o4, lse4, s, ws)
    assert B.device_status(ws) == (0, 0)
    assert torch.equal(o4, o2) and torch.equal(lse4, lse2)
    o3, lse3, res = fa.forward(q, k, v, causal=True, residual=True)
    dq, dk, dv = fa.backward(q, k, v, o3, lse3, do, causal=True, o_residual=res)
    torch.cuda.synchronize()
    dq_ref, dk_ref, dv_ref = A.attention_backward(x["q"], x["k"], x["v"], x["do"], s.scale, True)
    for g, r, n in ((dq, dq_ref, "dQ"), (dk, dk_ref, "dK"), (dv, dv_ref, "dV")):
        assert_grad(g, r, n + " after the timeout")
    assert np.array_equal(f64(o3), f64(o2))
