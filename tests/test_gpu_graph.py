"""The C-ABI calls inside a captured CUDA graph: a training step (forward, whose
launch overlaps its set-up with the header-clearing kernel before it, then the
backward) and a decode, captured once and replayed on new inputs copied into the
captured buffers, equal bit for bit to the same calls made eagerly, and to the
fp64 oracle within the usual bounds."""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import binding as B
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_training_step_in_a_graph_equals_eager():
    Bn, Hq, Hkv, N, d = 1, 4, 2, 1000, 128
    s = B.shape(Bn, Hq, Hkv, N, N, d, None, True)
    lib = fa.library()
    sets = [inputs.shape_inputs(Bn, Hq, Hkv, N, N, d, seed=40 + i) for i in range(3)]
    x = {k: sets[0][k].to(DEV) for k in ("q", "k", "v", "do")}  # the captured buffers
    nan = float("nan")  # outputs start as NaN: every element must be written
    o, res = torch.full_like(x["q"], nan), torch.full_like(x["q"], nan)
    lse = torch.full((Bn, Hq, N), nan, dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.full_like(x["q"], nan), torch.full_like(x["k"], nan), torch.full_like(x["v"], nan)
    wsf = torch.zeros(lib.fa_fwd_workspace_size(ctypes.byref(s)), dtype=torch.uint8, device=DEV)
    wsb = torch.zeros(lib.fa_bwd_workspace_size(ctypes.byref(s)), dtype=torch.uint8, device=DEV)

    def step():
        B.fa_fwd(x["q"], x["k"], x["v"], o, lse, s, wsf, res)
        B.fa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, s, wsb, res)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on the capturing stream (allocations, first-launch work)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for new in sets[1:]:
        for k in x:
            x[k].copy_(new[k].to(DEV))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        assert B.device_status(wsf) == (0, 0) and B.device_status(wsb) == (0, 0)
        step()  # the same calls, eagerly
        torch.cuda.synchronize()
        for a, b in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b)
        o_ref, lse_ref = A.attention_forward(new["q"], new["k"], new["v"], 1 / np.sqrt(d), True)
        assert_fwd(got[0], got[1], o_ref, lse_ref, "graph replay")


def test_decode_in_a_graph_equals_eager():
    Bn, Hq, Hkv, Nq, N, d = 2, 8, 2, 4, 3000, 128
    s = B.shape(Bn, Hq, Hkv, Nq, N, d)
    lib = fa.library()
    sets = [inputs.shape_inputs(Bn, Hq, Hkv, Nq, N, d, seed=60 + i, with_do=False) for i in range(2)]
    x = {k: sets[0][k].to(DEV) for k in ("q", "k", "v")}
    o = torch.full_like(x["q"], float("nan"))
    lse = torch.full((Bn, Hq, Nq), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(lib.fa_decode_workspace_size(ctypes.byref(s), 0), dtype=torch.uint8, device=DEV)
    call = lambda: B.fa_decode(x["q"], x["k"], x["v"], o, lse, s, 0, ws)  # noqa: E731
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    new = sets[1]
    for k in x:
        x[k].copy_(new[k].to(DEV))
    g.replay()
    torch.cuda.synchronize()
    got = (o.clone(), lse.clone())
    call()
    torch.cuda.synchronize()
    assert torch.equal(got[0], o) and torch.equal(got[1], lse)
    o_ref, lse_ref = A.attention_forward(new["q"], new["k"], new["v"], 1 / np.sqrt(d))
    assert_fwd(got[0], got[1], o_ref, lse_ref, "decode graph replay")
