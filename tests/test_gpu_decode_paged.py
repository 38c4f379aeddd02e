"""GPU parity of the paged, variable-length decode against the fp64 oracle (C ABI).

The cache is laid out in shuffled physical pages with spare pages; rows the
page tables do not reference hold junk (NaN in one test), which must never
reach the output.  Also: the key count recovered bit-exactly from LSE with
Q = 0, equality with the contiguous decode for an identity layout, device-side
reporting of bad lengths and page indices, and the full decode workload in
pages of 16 keys with ragged lengths, on sampled heads.  Shapes with Hkv a
multiple of 8 and pages of whole 16-row slices take the head-group kernel with
one CTA per 8 K/V heads; with Hkv a multiple of 4 or 2 and pages of 16-64 rows,
the same kernel with 4 or 2 heads per CTA (their warps merged per head); the
others the per-head kernel.
"""

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from parity import assert_fwd

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_pages(k, v, page_size, seed, spare=3, junk=7.0, device=DEV):
    """Contiguous [B, N, H, d] K/V -> shuffled pages [P, page_size, H, d] and an int32 table."""
    B, N, H, d = k.shape
    npb = -(-N // page_size)
    pages = B * npb + spare
    gen = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(pages, generator=gen).to(device)
    kc = torch.full((pages, page_size, H, d), junk, dtype=torch.bfloat16, device=device)
    vc = torch.full((pages, page_size, H, d), junk, dtype=torch.bfloat16, device=device)
    pad = npb * page_size - N
    kp = torch.nn.functional.pad(k.to(device), (0, 0, 0, 0, 0, pad), value=junk).reshape(B * npb, page_size, H, d)
    vp = torch.nn.functional.pad(v.to(device), (0, 0, 0, 0, 0, pad), value=junk).reshape(B * npb, page_size, H, d)
    used = perm[:B * npb]
    kc[used] = kp
    vc[used] = vp
    table = torch.full((B, npb + 2), -1, dtype=torch.int32, device=device)   # trailing entries: never read
    table[:, :npb] = used.reshape(B, npb).to(torch.int32)
    return kc, vc, table


def run(q, kc, vc, table, lens, max_len, S=0):
    o, lse = fa.decode_paged(q, kc, vc, table, lens, max_seqlen=max_len, num_splits=S)
    torch.cuda.synchronize()
    return o, lse


CASES = [
    # B, Hq, Hkv, Nq, lengths, d, page_size, splits
    (2, 8, 2, 4, [1000, 357], 128, 16, 0),      # 16 packed rows, pages smaller than a tile
    (3, 4, 1, 1, [1, 129, 2048], 64, 64, 0),
    (2, 16, 4, 4, [5000, 4097], 128, 256, 5),   # pages holding two tiles
    (1, 8, 8, 2, [128], 64, 128, 0),
    (4, 32, 8, 4, [300, 1, 2000, 777], 128, 32, 3),
    (2, 4, 2, 1, [4500, 20], 128, 16, 9),       # more splits than the short sequence has stages
    # K/V heads in groups of 8 (one CTA per group, 16-key page slices)
    (2, 16, 8, 2, [1000, 333], 64, 16, 0),
    (3, 8, 8, 1, [17, 1, 640], 128, 16, 0),
    (1, 32, 16, 1, [2049], 128, 256, 5),         # two head groups, pages of two tiles
    (2, 64, 16, 4, [700, 1500], 128, 32, 40),    # 16 packed rows, more splits than needed
    # 4 or 2 K/V heads per CTA (pages of 16-64 rows): 32- or 64-key stages, warps merged per head
    (2, 16, 4, 2, [3000, 77], 128, 32, 0),       # four heads, page = stage
    (1, 8, 4, 1, [2049], 64, 64, 3),             # four heads, two 32-row boxes per page
    (3, 12, 6, 2, [100, 1, 1500], 128, 16, 0),   # Hkv = 6: three groups of two, four boxes a stage
    (2, 4, 2, 8, [600, 1300], 64, 64, 2),        # two heads, 16 packed rows, page = stage
    (2, 8, 4, 2, [5000, 333], 128, 16, 50),      # more splits than the short sequence has stages
    (2, 8, 4, 1, [1000, 2000], 128, 16, 0),      # four heads, two 16-row boxes a stage
    (2, 4, 2, 2, [777, 64], 64, 16, 0),          # two heads, d = 64, four 16-row boxes a stage
    (1, 16, 4, 4, [1500], 64, 32, 2),            # four heads, d = 64, page = stage
    # more than 16 packed rows: the per-head kernel with two or four 16-row tiles
    (2, 16, 2, 4, [900, 2500], 128, 16, 0),      # 32 rows, pages of 16
    (2, 32, 8, 8, [300, 1200], 128, 16, 0),      # 32 rows with Hkv = 8 (no head groups past 16 rows)
    (1, 16, 2, 8, [4096], 64, 64, 3),            # 64 rows, d = 64
    (2, 8, 1, 6, [129, 2000], 128, 256, 0),      # 48 rows, pages of two tiles
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,lens,d,page,S", CASES)
def test_paged_decode_matches_oracle(B, Hq, Hkv, Nq, lens, d, page, S):
    N = max(lens)
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, N, d, seed=N + page + S, with_do=False)
    kc, vc, table = to_pages(x["k"], x["v"], page, seed=B * 7 + page)
    L = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = run(x["q"].to(DEV), kc, vc, table, L, N, S)
    o_ref, lse_ref = A.attention_decode_paged(x["q"], kc.float().cpu(), vc.float().cpu(), table.cpu().numpy(), lens,
                                              1 / np.sqrt(d))
    assert_fwd(o, lse, o_ref, lse_ref, f"paged {B}x{Hq}/{Hkv}x{Nq} lens={lens} d={d} page={page} S={S}")


@pytest.mark.parametrize("Hkv,page", [(2, 32), (8, 16), (4, 64), (1, 16)])
def test_nan_in_unreferenced_rows_never_reaches_the_output(Hkv, page):
    B, Hq, Nq, d = 3, 8, 2, 128
    lens = [77, 1, 300]
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, max(lens), d, seed=5, with_do=False)
    kc, vc, table = to_pages(x["k"], x["v"], page, seed=11, junk=float("nan"))
    L = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = run(x["q"].to(DEV), kc, vc, table, L, max(lens))
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    o_ref, lse_ref = A.attention_decode_paged(x["q"], kc.float().cpu(), vc.float().cpu(), table.cpu().numpy(), lens,
                                              1 / np.sqrt(d))
    assert_fwd(o, lse, o_ref, lse_ref, "NaN junk")


@pytest.mark.parametrize("page,Hkv", [(16, 2), (64, 2), (128, 2), (16, 8), (32, 4)])
def test_zero_query_counts_each_sequence_keys_exactly(page, Hkv):
    lens = [1, 127, 128, 129, 1000, 4095]
    B, Hq, Nq, d = len(lens), 2 * Hkv, 1, 64
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, max(lens), d, seed=page, with_do=False)
    kc, vc, table = to_pages(x["k"], x["v"], page, seed=page)
    q = torch.zeros(B, Nq, Hq, d, dtype=torch.bfloat16, device=DEV)
    o, lse = run(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32, device=DEV), max(lens), 3)
    counts = torch.round(torch.exp(lse.double())).long().cpu()
    expect = torch.tensor(lens).view(B, 1, 1).expand(B, Hq, Nq)
    assert torch.equal(counts, expect), (counts, expect)


def test_identity_layout_equals_contiguous_decode():
    B, Hq, Hkv, Nq, N, d = 2, 8, 2, 4, 4096, 128
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, N, d, seed=21, with_do=False)
    q, k, v = x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV)
    o_c, lse_c = fa.decode(q, k, v, num_splits=6)
    kc = k.reshape(B * (N // 128), 128, Hkv, d)
    vc = v.reshape(B * (N // 128), 128, Hkv, d)
    table = torch.arange(B * (N // 128), dtype=torch.int32, device=DEV).reshape(B, N // 128)
    o_p, lse_p = run(q, kc, vc, table, torch.full((B,), N, dtype=torch.int32, device=DEV), N, 6)
    assert torch.equal(o_p, o_c) and torch.equal(lse_p, lse_c)


@pytest.mark.parametrize("Hq,Hkv,page", [(4, 1, 64), (8, 8, 16), (8, 2, 32)])
def test_bad_lengths_and_pages_are_reported_not_faulted(Hq, Hkv, page):
    B, Nq, d, N = 3, 1, 64, 512
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, N, d, seed=3, with_do=False)
    kc, vc, table = to_pages(x["k"], x["v"], page, seed=3)
    q = x["q"].to(DEV)
    s = fa.binding.shape(B, Hq, Hkv, Nq, N, d)
    lib = fa.library()
    import ctypes

    def call(lens, tab):
        ws = torch.zeros(lib.fa_decode_paged_workspace_size(ctypes.byref(s), 0, page), dtype=torch.uint8, device=DEV)
        o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=DEV)
        fa.binding.fa_decode_paged(q, kc, vc, tab, torch.tensor(lens, dtype=torch.int32, device=DEV), o, lse, s, 0,
                                   ws)
        return fa.binding.device_status(ws), o, lse

    (rc, st), o, _ = call([N, 200, 1], table)
    assert rc == 0 and st == 0
    (rc, st), o, _ = call([N, 0, N + 5], table)      # a length below 1 and one above Nk
    assert rc == 1 and st & 0x100
    assert torch.isfinite(o[0]).all()
    bad = table.clone()
    bad[1, 1] = kc.shape[0] + 10                      # a page index out of range
    (rc, st), o, _ = call([N, 200, 1], bad)
    assert rc == 1 and st & 0x100
    torch.cuda.synchronize()


@pytest.mark.slow
@pytest.mark.parametrize("w", [inputs.DECODE_Q1, inputs.DECODE_Q4], ids=lambda w: w.name)
def test_full_decode_paged16_ragged_sampled(w):
    x = inputs.make(w, device=DEV, with_do=False)
    q, k, v = x["q"], x["k"], x["v"]
    gen = torch.Generator(device="cpu").manual_seed(17)
    lens = torch.randint(w.Nk // 2, w.Nk + 1, (w.B,), generator=gen)
    kc, vc, table = to_pages(k, v, 16, seed=17)
    o, lse = run(q, kc, vc, table, lens.to(torch.int32).to(DEV), w.Nk)
    del kc, vc
    g = w.Hq // w.Hkv
    for b, kvh in [(0, 0), (w.B // 2, 3), (w.B - 1, w.Hkv - 1)]:
        L = int(lens[b])
        hs = slice(kvh * g, (kvh + 1) * g)
        qs = q[b:b + 1, :, hs].cpu()
        ks, vs = k[b:b + 1, :L, kvh:kvh + 1].cpu(), v[b:b + 1, :L, kvh:kvh + 1].cpu()
        o_ref, lse_ref = A.attention_forward(qs, ks, vs, w.scale)
        assert_fwd(o[b:b + 1, :, hs], lse[b:b + 1, hs], o_ref, lse_ref, f"{w.name} paged16 b{b} kvh{kvh} L={L}")
    assert torch.isfinite(o).all()
