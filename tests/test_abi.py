"""The C-ABI library loads, exports every declared symbol, and its host plans
equal the oracle's plans exactly (no GPU needed: no compute call is made)."""

import ctypes
import os
import re

import pytest

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300.binding import SIGNATURES, FaShape, FaTensor, shape
from oracle import plan as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.library_path()):
        from exact_io_aware_21_gb300 import build

        build.build()
    return fa.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(fa_[a-z0-9_]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(SIGNATURES), "binding signatures must mirror the header"


def test_strerror(lib):
    assert lib.fa_strerror(0) == b"ok"
    for code in range(1, 8):
        assert len(lib.fa_strerror(code)) > 5


def S(B, Hq, Hkv, Nq, Nk, d=128, causal=False):
    return ctypes.byref(shape(B, Hq, Hkv, Nq, Nk, d, causal=causal))


@pytest.mark.parametrize("N", [128, 200, 1000, 4096])
@pytest.mark.parametrize("causal", [False, True])
def test_tile_classes_match_oracle(lib, N, causal):
    want = P.tile_classes(N, N, 128, 128, causal)
    for i, row in enumerate(want):
        for j, c in enumerate(row):
            assert lib.fa_tile_class(S(1, 1, 1, N, N, causal=causal), i, j) == c


@pytest.mark.parametrize("N,left,right,causal", [(1000, 100, 50, False), (777, 300, -1, True), (512, 0, 0, False),
                                                 (640, 128, 128, False), (300, 1000, 3, True), (4096, 1024, 0, True),
                                                 (640, 128, -1, False), (1000, -1, 200, False)])
def test_window_tile_classes_match_oracle(lib, N, left, right, causal):
    s = ctypes.byref(shape(1, 1, 1, N, N, 64, causal=causal, window=(left, right)))
    nt = -(-N // 128)
    for i in range(nt):
        for j in range(nt):
            want = P.window_tile_class(i * 128, min(N, i * 128 + 128), j * 128, min(N, j * 128 + 128), left, right,
                                       causal)
            assert lib.fa_tile_class(s, i, j) == want, (i, j)


def test_window_needs_square_shape(lib):
    s = shape(1, 1, 1, 100, 200, 64, window=(10, 10))
    assert lib.fa_tile_class(ctypes.byref(s), 0, 0) == -1
    s.window = 2
    s.Nk = 100
    assert lib.fa_tile_class(ctypes.byref(s), 0, 0) == -1


def test_noncausal_rectangular_classes(lib):
    assert lib.fa_tile_class(S(1, 1, 1, 100, 700), 0, 5) == P.FULL
    assert lib.fa_tile_class(S(1, 1, 1, 100, 700), 0, 6) == -1   # out of range


def units(lib, kind, s, n):
    out = []
    b, x, y = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    fn = getattr(lib, f"fa_{kind}_unit")
    for i in range(n):
        assert fn(s, i, ctypes.byref(b), ctypes.byref(x), ctypes.byref(y)) == 0
        out.append((b.value, x.value, y.value))
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(2, 4, 2, 128), (2, 4, 4, 300), (1, 8, 2, 1000), (2, 16, 16, 4096),
                                        (1, 32, 8, 8192)])
def test_unit_orders_match_oracle(lib, causal, B, Hq, Hkv, N):
    s = S(B, Hq, Hkv, N, N, causal=causal)
    n = lib.fa_fwd_num_units(s)
    assert units(lib, "fwd", s, n) == P.fwd_unit_order(B, Hq, N, N, causal)
    n = lib.fa_dkdv_num_units(s)
    assert units(lib, "dkdv", s, n) == P.dkdv_unit_order(B, Hkv, N, N, causal)
    n = lib.fa_dq_num_units(s)
    assert units(lib, "dq", s, n) == P.dq_unit_order(B, Hq, N, N, causal)


@pytest.mark.parametrize("Nk", [1, 127, 128, 129, 1000, 131072])
@pytest.mark.parametrize("req", [1, 3, 19, 64])
def test_decode_split_ranges_match_oracle(lib, Nk, req):
    s = S(8, 32, 8, 1, Nk)
    want = P.decode_splits(Nk, req)
    assert lib.fa_decode_num_splits(s, req) == len(want)
    a, b = ctypes.c_int(), ctypes.c_int()
    got = []
    for i in range(len(want)):
        assert lib.fa_decode_split_range(s, req, i, ctypes.byref(a), ctypes.byref(b)) == 0
        got.append((a.value, b.value))
    assert got == want
    assert lib.fa_decode_split_range(s, req, len(want), ctypes.byref(a), ctypes.byref(b)) != 0


def test_decode_auto_splits_positive(lib):
    n = lib.fa_decode_num_splits(S(8, 32, 8, 4, 131072), 0)
    assert 1 <= n <= 1024


FAKE = 0x10000  # never dereferenced: argument checks fail first


def tens(ptr=FAKE, sb=8 * 1024, sn=8 * 16, sh=8 * 2):
    return ctypes.byref(FaTensor(ptr, sb, sn, sh))


@pytest.mark.parametrize("bad", [
    dict(Hq=3, Hkv=2), dict(d=96), dict(B=0), dict(Nq=0), dict(causal=True, Nq=10, Nk=20), dict(scale=0.0),
    dict(scale=float("nan")), dict(scale=-1.0)])
def test_invalid_shapes_rejected_before_any_gpu_work(lib, bad):
    kw = dict(B=1, Hq=2, Hkv=2, Nq=16, Nk=16, d=64, causal=False, scale=None)
    kw.update(bad)
    s = shape(**kw)
    if bad.get("scale", 1.0) != bad.get("scale", 1.0) or "scale" in bad:
        s.scale = bad["scale"]
    rc = lib.fa_fwd(tens(), tens(), tens(), tens(), FAKE, None, ctypes.byref(s), FAKE, 1 << 20, None)
    assert rc == 1  # FA_ERR_INVALID


def test_misaligned_and_workspace_errors(lib):
    s = ctypes.byref(shape(1, 2, 2, 16, 16, 64))
    assert lib.fa_fwd(tens(FAKE + 2), tens(), tens(), tens(), FAKE, None, s, FAKE, 1 << 20, None) == 2
    assert lib.fa_fwd(tens(sn=12), tens(), tens(), tens(), FAKE, None, s, FAKE, 1 << 20, None) == 2
    assert lib.fa_fwd(tens(), tens(), tens(), tens(), FAKE, None, s, FAKE, 8, None) == 3
    assert lib.fa_fwd(tens(), tens(), tens(), tens(), FAKE, tens(FAKE + 4), s, FAKE, 1 << 20, None) == 2
    assert lib.fa_fwd(tens(), tens(), tens(), tens(), None, None, s, FAKE, 1 << 20, None) == 1
    assert lib.fa_fwd(None, tens(), tens(), tens(), FAKE, None, s, FAKE, 1 << 20, None) == 1
    # bwd_part: unknown part
    assert lib.fa_bwd_part(3, tens(), tens(), tens(), tens(), FAKE, None, tens(), tens(), tens(), tens(), s, FAKE,
                           1 << 20, None) == 1
    # decode: more than 64 packed rows (four 16-row tiles) are rejected
    sd = shape(1, 80, 1, 1, 100, 64)
    assert lib.fa_decode(tens(), tens(), tens(), tens(), FAKE, ctypes.byref(sd), 1, FAKE, 1 << 30, None) == 1


@pytest.mark.parametrize("page_size,max_pages,table,lens", [
    (48, 64, FAKE, FAKE),      # neither 16/32/64 nor a multiple of 128
    (96, 64, FAKE, FAKE),
    (8, 256, FAKE, FAKE),
    (16, 4, FAKE, FAKE),       # 4 pages of 16 cannot hold Nk = 1000
    (16, 64, None, FAKE),      # no page table
    (16, 64, FAKE, None)])     # no lengths
def test_paged_decode_arguments_rejected_before_any_gpu_work(lib, page_size, max_pages, table, lens):
    sd = ctypes.byref(shape(2, 8, 2, 4, 1000, 64))
    rc = lib.fa_decode_paged(tens(), tens(), tens(), table, max_pages, lens, 100, page_size, tens(), FAKE, sd, 0,
                             FAKE, 1 << 30, None)
    assert rc == 1  # FA_ERR_INVALID


def test_fp8_arguments_rejected_before_any_gpu_work(lib):
    s128 = ctypes.byref(shape(1, 2, 2, 256, 256, 128))
    s64 = ctypes.byref(shape(1, 2, 2, 256, 256, 64))
    u8 = lambda ptr=FAKE, sn=256: tens(ptr, sb=256 * 256, sn=sn, sh=128)  # noqa: E731

    def fwd8(q=None, s=s128, qs=FAKE, ws_bytes=1 << 20):
        return lib.fa_fwd_fp8(q or u8(), u8(), u8(), qs, FAKE, FAKE, tens(), FAKE, s, FAKE, ws_bytes, None)
    assert fwd8(s=s64) == 1                    # d = 128 only
    assert fwd8(q=u8(sn=264)) == 2             # code rows must be 16-byte multiples
    assert fwd8(q=u8(FAKE + 8)) == 2
    assert fwd8(qs=None) == 1
    assert fwd8(ws_bytes=8) == 3

    def quant(d=128, rows=128, out=None, scales=FAKE, ws_bytes=1 << 20, x=None):
        return lib.fa_quantize_fp8(x or tens(), 1, 256, 2, d, rows, None, out or u8(), scales, FAKE, ws_bytes, None)
    assert quant(d=96) == 1
    assert quant(rows=64) == 1
    assert quant(scales=None) == 1
    assert quant(out=u8(sn=136)) == 2
    assert quant(x=tens(FAKE + 2)) == 2
    assert quant(ws_bytes=16) == 3
    assert lib.fa_quantize_fp8_workspace_size(2, 3) >= 256 + 2 * 3 * 4
    assert lib.fa_quantize_fp8_workspace_size(0, 3) == 0


def test_varlen_arguments_rejected_before_any_gpu_work(lib):
    s = ctypes.byref(shape(3, 2, 2, 500, 500, 64, causal=True))          # B sequences, packed totals
    sw = ctypes.byref(shape(3, 2, 2, 500, 500, 64, window=(10, 0)))
    pk = lambda ptr=FAKE: tens(ptr, sb=0, sn=2 * 64, sh=64)  # noqa: E731

    def fwd(cq=FAKE, ck=FAKE, mq=300, mk=300, sh=s):
        return lib.fa_fwd_varlen(pk(), pk(), pk(), cq, ck, mq, mk, pk(), FAKE, None, sh, FAKE, 1 << 20, None)
    assert fwd(cq=None) == 1 and fwd(ck=None) == 1
    assert fwd(mq=0) == 1 and fwd(mk=501) == 1                           # longest length outside [1, total]
    assert fwd(sh=sw) == 1                                              # no window with packing
    assert lib.fa_fwd_varlen(pk(), pk(), pk(), FAKE, FAKE, 300, 300, pk(), FAKE, None, s, FAKE, 64, None) == 3
    assert lib.fa_fwd_varlen_workspace_size(s, 300) >= 256 + 4 * (4 + 2 + 1 + 3)
    assert lib.fa_fwd_varlen_workspace_size(s, 0) == 0
    assert lib.fa_bwd_varlen_workspace_size(s, 300) > lib.fa_bwd_varlen_workspace_size(s, 100) > 0
    assert lib.fa_bwd_varlen(pk(), pk(), pk(), FAKE, FAKE, 0, 300, pk(), FAKE, None, pk(), pk(), pk(), pk(), s, FAKE,
                             1 << 30, None) == 1


def test_blocksparse_arguments_rejected_before_any_gpu_work(lib):
    s = ctypes.byref(shape(1, 2, 2, 1000, 1000, 64))

    def fwd(rp=FAKE, ci=FAKE, nnz=5, sh=s):
        return lib.fa_fwd_blocksparse(tens(), tens(), tens(), rp, ci, nnz, tens(), FAKE, None, sh, FAKE, 1 << 20,
                                      None)
    assert fwd(rp=None) == 1 and fwd(ci=None) == 1 and fwd(nnz=-1) == 1
    assert fwd(sh=ctypes.byref(shape(1, 2, 2, 1000, 131200, 64))) == 1      # more than 1024 key tiles
    assert fwd(sh=ctypes.byref(shape(1, 2, 2, 1000, 1000, 64, window=(5, 5)))) == 1
    big = ctypes.byref(shape(1, 2, 2, 131200, 1000, 64))
    assert lib.fa_bwd_blocksparse(tens(), tens(), tens(), FAKE, FAKE, 5, tens(), FAKE, None, tens(), tens(), tens(),
                                  tens(), big, FAKE, 1 << 30, None) == 1
    assert lib.fa_bwd_blocksparse_workspace_size(s, 400) > lib.fa_bwd_blocksparse_workspace_size(s, 0) > 0


def test_workspace_sizes(lib):
    s = S(2, 16, 16, 4096, 4096, causal=True)
    assert lib.fa_fwd_workspace_size(s) >= 256
    assert lib.fa_bwd_workspace_size(s) >= 256 + 2 * 2 * 16 * 4096 * 4
    sd = S(8, 32, 8, 4, 131072)
    n = lib.fa_decode_num_splits(sd, 19)
    assert lib.fa_decode_workspace_size(sd, 19) >= 256 + 8 * 32 * 4 * n * (128 + 1) * 4
    lo, oo = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.fa_decode_partials_layout(sd, 19, ctypes.byref(lo), ctypes.byref(oo)) == 0
    assert lo.value == 256 and oo.value >= lo.value + 8 * 32 * 4 * n * 4


def test_binding_rejects_non_cuda_tensors():
    import torch

    with pytest.raises(fa.FAError):
        fa.binding.tdesc(torch.zeros(1, 2, 2, 64, dtype=torch.bfloat16))


# ------------------------------------------------------------------ block-sparse dK/dV plan bounds
def _segment_rule(M, causal, heads, g, P=152, min_seg=32):
    """The dK/dV segment rule of the block-sparse backward: per key tile n = g x
    (query tiles listing it, under causal those at or below the diagonal);
    seg = max(32, ceil(heads * sum(n) / P)); a tile with n > seg becomes
    ceil(n / seg) segments (else one), each segment of a split tile a partial tile."""
    nqt, nkt = len(M), len(M[0])
    n = [g * sum(1 for i in range(nqt) if M[i][j] and (not causal or j <= i)) for j in range(nkt)]
    seg = max(min_seg, -(-heads * sum(n) // P))
    nseg = [(-(-x // seg) if x > seg else 1) for x in n]
    return sum(nseg), heads * sum(k for k in nseg if k > 1)


def test_block_sparse_plan_fits_its_bounds(lib):
    """On random tables, dense rows, one global column and a full table, the plan
    holds fewer than nkt + 2P segments per head group and fewer partial tiles
    (all heads) than the workspace's pool: min(2P, ceil(heads * g * nnz / 16))."""
    import random

    rng = random.Random(5)
    cases = []
    for _ in range(300):
        nqt, nkt = rng.randint(1, 96), rng.randint(1, 96)
        dens = rng.choice([0.02, 0.1, 0.5, 1.0])
        M = [[rng.random() < dens for _ in range(nkt)] for _ in range(nqt)]
        if rng.random() < 0.3:
            for i in range(nqt):
                M[i][0] = True                      # a global column
        cases.append((M, rng.random() < 0.5 and nqt == nkt, rng.choice([1, 2, 8, 32]), rng.choice([1, 2, 4, 8])))
    cases.append(([[True] * 1024 for _ in range(1024)], False, 1, 8))   # the largest table, full
    cases.append(([[j == 0 or j == i for j in range(512)] for i in range(512)], True, 64, 4))
    for M, causal, heads, g in cases:
        nnz = sum(map(sum, M))
        segs, slots = _segment_rule(M, causal, heads, g)
        assert segs < len(M[0]) + 2 * 152
        assert slots <= min(2 * 152, -(-heads * g * nnz // 16))


def test_paged_decode_workspace_covers_its_splits(lib):
    """The paged decode's workspace: head-group shapes (8 K/V heads per CTA when Hkv %
    8 == 0 and pages are whole 16-row slices; 4 or 2 when pages hold 16-64 rows) size
    the partials for their own split count, capped at one stage (128 / heads-per-CTA
    keys) each; the others match the contiguous decode's."""
    size = lib.fa_decode_paged_workspace_size
    hdr = 256

    def parts(B, Hq, Nq, S, d=128):
        rows = B * Hq * Nq * S
        up = lambda x: -(-x // 256) * 256  # noqa: E731
        return hdr + up(rows * 4) + up(rows * d * 4)

    s8 = S(8, 32, 8, 1, 131072)
    assert size(s8, 5, 16) == parts(8, 32, 1, 5)                  # explicit splits, head groups
    assert size(s8, 5000, 16) == parts(8, 32, 1, 5000)
    assert size(S(1, 8, 8, 1, 1000), 100, 16) == parts(1, 8, 1, 63)  # capped at one 16-key slice each
    s2 = S(2, 8, 2, 4, 4096)
    assert size(s2, 5, 16) == parts(2, 8, 4, 5)                    # two heads per CTA
    assert size(S(1, 8, 2, 1, 1000), 100, 64) == parts(1, 8, 1, 16)  # capped at 64-key stages
    assert size(S(1, 8, 4, 1, 1000), 100, 32) == parts(1, 8, 1, 32)  # four heads: 32-key stages
    assert size(s2, 0, 128) == lib.fa_decode_workspace_size(s2, 0)  # pages of whole tiles: per-head kernel
    s1 = S(2, 8, 1, 2, 4096)
    assert size(s1, 0, 16) == lib.fa_decode_workspace_size(s1, 0)  # one K/V head: per-head kernel
    assert size(s8, 3, 48) == lib.fa_decode_workspace_size(s8, 3)  # pages not of whole 16-row slices
    assert size(S(1, 8, 8, 1, 0), 0, 16) == 0                      # invalid shape


def _pair_products(N, p):
    """Tensor-core products of causal forward unit p: two per key tile visited by each of
    its query tiles (S and P V), counted from the causal tile classes."""
    nt = P.cdiv(N, 128)
    n = 0
    for t in (2 * p, 2 * p + 1):
        if t < nt:
            n += sum(1 for j in range(nt)
                     if P.causal_tile_class(t * 128, min(N, t * 128 + 128), j * 128, min(N, j * 128 + 128)) != P.SKIP)
    return 2 * n


@pytest.mark.parametrize("B,Hq,N,d,grid", [(2, 16, 4096, 128, 152), (1, 32, 8192, 128, 152), (2, 4, 1000, 128, 16),
                                           (1, 6, 1100, 64, 24), (3, 5, 3000, 64, 152)])
def test_fwd_schedule_is_a_balanced_partition(lib, B, Hq, N, d, grid):
    """The static schedule of a causal forward runs every unit exactly once, each CTA's
    units longest first, and its largest CTA load (products plus a fixed 16 x 128 / d per
    unit) is no worse than handing the units out longest first."""
    s = S(B, Hq, Hq, N, N, d=d, causal=True)
    n = lib.fa_fwd_num_units(s)
    grid = min(grid, n)
    start = (ctypes.c_int * (grid + 1))()
    ord_ = (ctypes.c_int * n)()
    assert lib.fa_fwd_schedule(s, grid, start, ord_) == 0
    st, od = list(start), list(ord_)
    assert st[0] == 0 and st[-1] == n and all(a <= b for a, b in zip(st, st[1:]))
    assert sorted(od) == list(range(n))
    cost = []
    for u in range(n):
        b, h, p = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        assert lib.fa_fwd_unit(s, u, ctypes.byref(b), ctypes.byref(h), ctypes.byref(p)) == 0
        cost.append(_pair_products(N, p.value) + 16 * 128 // d)
    loads = []
    for c in range(grid):
        mine = [cost[u] for u in od[st[c]:st[c + 1]]]
        assert mine == sorted(mine, reverse=True)
        loads.append(sum(mine))
    assert max(loads) <= max(P.greedy_loads(cost, grid, True))
    assert max(loads) >= sum(cost) / grid


@pytest.mark.parametrize("B,H,N,d,sms", [(4, 16, 2048, 64, 152), (1, 8, 2048, 128, 152), (2, 2, 513, 64, 152),
                                         (1, 2, 200, 128, 152), (1, 16, 4096, 128, 152), (1, 1, 256, 64, 152),
                                         (3, 5, 3000, 64, 16), (1, 4, 8192, 128, 152)])
def test_fwd_split_plan(lib, B, H, N, d, sms):
    """The unmasked forward's key-split plan: only the last wave's units are split (all of
    them when there are fewer than SMs), into 2-4 parts of at least two key tiles, and the
    split wave then fits on the SMs, so the launch's length in unit times drops from
    ceil(U / sms) to floor(U / sms) + 1 / nsplit."""
    s = S(B, H, H, N, N, d=d)
    U = lib.fa_fwd_num_units(s)
    nk = -(-N // 128)
    s0, ns = ctypes.c_int(), ctypes.c_int()
    assert lib.fa_fwd_split_plan(s, sms, ctypes.byref(s0), ctypes.byref(ns)) == 0
    R = U % sms if U >= sms else U
    if ns.value == 1:
        assert s0.value == U
        assert R == 0 or min(sms // R, 4, nk // 2) < 2
        return
    assert s0.value == U - R and 2 <= ns.value <= 4 and ns.value * 2 <= nk
    assert R * ns.value <= sms                        # the split wave fits on the SMs
    assert ns.value == min(sms // R, 4, nk // 2)
    waves_before = -(-U // sms)
    assert U // sms + 1 / ns.value < waves_before     # shorter in unit times


def test_fwd_split_plan_only_without_a_mask(lib):
    s0, ns = ctypes.c_int(), ctypes.c_int()
    assert lib.fa_fwd_split_plan(S(1, 2, 2, 1000, 1000, causal=True), 152, ctypes.byref(s0), ctypes.byref(ns)) == 1
    windowed = ctypes.byref(shape(1, 2, 2, 1000, 1000, 128, window=(5, 5)))
    assert lib.fa_fwd_split_plan(windowed, 152, ctypes.byref(s0), ctypes.byref(ns)) == 1


def test_fwd_schedule_only_for_causal(lib):
    start = (ctypes.c_int * 153)()
    ord_ = (ctypes.c_int * 4096)()
    assert lib.fa_fwd_schedule(S(2, 16, 16, 4096, 4096), 152, start, ord_) == 1
