"""fa_decode_noalloc: split-KV decode for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: an inference server that
reserves all device memory for its own pool at start-up, or a plug-in that
only receives the call's tensors.  fa_decode_noalloc gives them the same
decode as fa_decode, with its scratch in a fixed array inside the library.
These tests call both entry points through the C ABI on the same inputs and
require the outputs to agree within the parity tolerances, and both to match
the fp64 oracle, on two calls in a row (the second call reuses the array the
first one left behind); after each call the array's status header, read with
fa_decode_noalloc_status, must report no error.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes when run alone.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from exact_io_aware_21_gb300.binding import check, tdesc
from oracle import attention as A
from parity import assert_fwd

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def noalloc(q, k, v, num_splits):
    s = fa.binding._dims(q, k, None, False)
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((s.B, s.Hq, s.Nq), float("nan"), dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    check(fa.library().fa_decode_noalloc(tdesc(q), tdesc(k), tdesc(v), tdesc(o), lse.data_ptr(), ctypes.byref(s),
                                         int(num_splits), stream))
    bits = ctypes.c_int(-1)
    rc = fa.library().fa_decode_noalloc_status(stream, ctypes.byref(bits))
    assert rc == 0 and bits.value == 0, f"status {bits.value:#x}"
    return o, lse


def draw(B, Hq, Hkv, Nq, Nk, seed):
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, 128, seed=seed, with_do=False)
    return x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV)


@pytest.mark.parametrize("num_splits", [5, 0])
def test_matches_fa_decode_on_two_calls_in_a_row(num_splits):
    shapes = [(2, 8, 2, 4, 3000, 11), (1, 4, 1, 1, 20000, 12)]
    for B, Hq, Hkv, Nq, Nk, seed in shapes:   # two calls in a row, different problems
        q, k, v = draw(B, Hq, Hkv, Nq, Nk, seed)
        o_ref, lse_ref = fa.decode(q, k, v, num_splits=num_splits)
        o, lse = noalloc(q, k, v, num_splits)
        assert_fwd(o, lse, o_ref, lse_ref, f"noalloc vs fa_decode {B}x{Hq}/{Hkv}x{Nq}x{Nk}")
        o_or, lse_or = A.attention_forward(q.cpu(), k.cpu(), v.cpu(), 1 / np.sqrt(128))
        assert_fwd(o, lse, o_or, lse_or, f"noalloc vs the oracle {B}x{Hq}/{Hkv}x{Nq}x{Nk}")
    # and the same problem twice: identical results
    q, k, v = draw(2, 8, 2, 4, 3000, 11)
    a = noalloc(q, k, v, num_splits)
    b = noalloc(q, k, v, num_splits)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_rejects_problems_beyond_the_fixed_scratch():
    lib = fa.library()
    cap = lib.fa_decode_noalloc_max_bytes()
    assert cap == 8 << 20
    B, Hq, Hkv, Nq, Nk = 8, 32, 8, 4, 131072
    s = fa.binding.shape(B, Hq, Hkv, Nq, Nk, 128)
    splits = 64                                  # needs far more than the array holds
    assert lib.fa_decode_workspace_size(ctypes.byref(s), splits) > cap
    q = torch.zeros(B, Nq, Hq, 128, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(B, 256, Hkv, 128, dtype=torch.bfloat16, device=DEV)   # never read: rejected first
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=DEV)
    rc = lib.fa_decode_noalloc(tdesc(q), tdesc(kv), tdesc(kv), tdesc(o), lse.data_ptr(), ctypes.byref(s), splits,
                               None)
    assert rc == 8 and b"scratch" in lib.fa_strerror(rc)
