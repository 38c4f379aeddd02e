"""GPU parity of the block-sparse forward and backward against the fp64 oracle,
through fa_fwd_blocksparse and fa_bwd_blocksparse.

Covers random tables over ragged shapes (causal and not, grouped heads, d = 64
and 128, rows with no listed tile, key tiles no row lists), every tile listed
against the dense kernels (bit for bit), a sliding-window + global-token
pattern at N = 8192 on sampled query tiles, the residual, tables that break
the rules (reported), key tiles long enough for the dK/dV plan to split (plan,
determinism, parity) and the local + global pattern at N = 16384 sampled."""

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
    fa.library().fa_set_wait_timeout_ns(10_000_000_000)


def csr(M):
    rows = [np.flatnonzero(r) for r in M]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.concatenate(rows).astype(np.int32) if sum(len(r) for r in rows) else np.zeros(0, np.int32)
    return rp, ci


def run(x, M, causal, scale, residual=False):
    rp, ci = csr(M)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out = fa.forward_blocksparse(q, k, v, torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV),
                                 causal=causal, scale=scale, residual=residual)
    torch.cuda.synchronize()
    return out, rp, ci


CASES = [  # B, Hq, Hkv, Nq, Nk, d, causal, density
    (1, 2, 1, 640, 900, 64, False, 0.4),
    (2, 4, 2, 1000, 1000, 128, True, 0.5),
    (1, 2, 2, 384, 384, 128, False, 0.3),
    (1, 8, 2, 2048, 2048, 128, True, 0.25),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,density", CASES)
def test_random_tables(B, Hq, Hkv, Nq, Nk, d, causal, density):
    g = np.random.default_rng(Nq + Nk + d)
    nqt, nkt = -(-Nq // 128), -(-Nk // 128)
    M = g.random((nqt, nkt)) < density
    M[np.arange(nqt), np.arange(nqt) % nkt] = True              # every query tile lists a tile ...
    M[1] = False                                               # ... but one
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq + d, with_do=False)
    scale = 1 / np.sqrt(d)
    (o, lse), rp, ci = run(x, M, causal, scale)
    o_ref, lse_ref = A.attention_blocksparse_forward(x["q"], x["k"], x["v"], rp, ci, scale, causal)
    seen = np.isfinite(lse_ref[0, 0])
    tag = f"blocksparse {B}x{Hq}/{Hkv} {Nq}x{Nk} d={d} causal={causal}"
    assert_fwd(o[:, seen], lse[:, :, seen], o_ref[:, seen], lse_ref[:, :, seen], tag)
    assert not f64(o[:, ~seen]).any() and np.all(np.isneginf(f64(lse[:, :, ~seen]))), tag


@pytest.mark.parametrize("causal,d", [(False, 64), (True, 128)])
def test_every_tile_listed_equals_the_dense_kernel(causal, d):
    """With every tile listed the block-sparse kernel does the dense kernel's work:
    bit for bit where the dense call runs whole units (causal).  Without a mask the
    dense call splits this small grid's units along the keys and merges the parts
    by their LSE, so there both are held to the exact result instead."""
    N = 1000
    x = inputs.shape_inputs(2, 4, 2, N, N, d, seed=3, with_do=False)
    nt = -(-N // 128)
    (o, lse, res), _, _ = run(x, np.ones((nt, nt), bool), causal, 0.1, residual=True)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o2, lse2, res2 = fa.forward(q, k, v, causal=causal, scale=0.1, residual=True)
    torch.cuda.synchronize()
    if causal:
        assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(res, res2)
    else:
        o_ref, lse_ref = A.attention_forward(x["q"], x["k"], x["v"], 0.1, False)
        assert_fwd(o, lse, o_ref, lse_ref, "block-sparse, every tile listed", o_res=res)
        assert_fwd(o2, lse2, o_ref, lse_ref, "dense, key-split units", o_res=res2)


@pytest.mark.slow
def test_window_plus_global_pattern_sampled():
    """Each query tile lists its own tile, the two before it and tile 0 (a global
    prefix); causal; GQA 32/8 at N = 8192."""
    N, d = 8192, 128
    nt = N // 128
    M = np.zeros((nt, nt), bool)
    for i in range(nt):
        M[i, max(0, i - 2):i + 1] = True
        M[i, 0] = True
    w = inputs.Workload("bs", 1, 32, 8, N, N, d, True, seed=5)
    x = inputs.make(w, device=DEV, with_do=False)
    rp, ci = csr(M)
    o, lse = fa.forward_blocksparse(x["q"], x["k"], x["v"], torch.from_numpy(rp).to(DEV),
                                    torch.from_numpy(ci).to(DEV), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    q, k, v = (x[n][:, :, :].cpu() for n in ("q", "k", "v"))
    for qt in (0, 1, 37, nt - 1):
        rows = np.arange(qt * 128, (qt + 1) * 128)
        keys = np.concatenate([np.arange(j * 128, (j + 1) * 128) for j in np.flatnonzero(M[qt])])
        for h in (0, 13, 31):
            kv = h // 4
            qq, kk, vv = q[:, rows, h:h + 1], k[:, keys, kv:kv + 1], v[:, keys, kv:kv + 1]
            # causal within the gathered keys: key keys[j] visible to row rows[i] iff keys[j] <= rows[i]
            S = (f64(qq)[0, :, 0] @ f64(kk)[0, :, 0].T) * w.scale
            S = np.where(keys[None, :] <= rows[:, None], S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            o_ref = (E @ f64(vv)[0, :, 0]) / E.sum(axis=1, keepdims=True)
            lse_ref = m[:, 0] + np.log(E.sum(axis=1))
            assert_fwd(o[0, rows, h], lse[0, h, rows], o_ref, lse_ref, f"tile {qt} head {h}")


@pytest.mark.parametrize("table", ["decreasing", "out_of_range", "row_ptr_past_nnz"])
def test_tables_that_break_the_rules_are_reported(table):
    N = 384
    x = inputs.shape_inputs(1, 2, 2, N, N, 64, seed=1, with_do=False)
    rp = np.array([0, 2, 3, 4], np.int32)
    ci = np.array([0, 1, 1, 2], np.int32)
    if table == "decreasing":
        ci = np.array([1, 0, 1, 2], np.int32)
    elif table == "out_of_range":
        ci = np.array([0, 3, 1, 2], np.int32)
    else:
        rp = np.array([0, 2, 3, 9], np.int32)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    s = fa.binding._dims(q, k, None, False)
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 2, N), dtype=torch.float32, device=DEV)
    ws = torch.zeros(fa.library().fa_fwd_workspace_size(fa.binding.ctypes.byref(s)), dtype=torch.uint8, device=DEV)
    fa.fa_fwd_blocksparse(q, k, v, torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV), o, lse, s, ws)
    rc, st = fa.binding.device_status(ws)
    assert rc == 1 and st == 0x100


# ------------------------------------------------------------------ backward
from parity import assert_grad  # noqa: E402


def run_bwd(x, M, causal, scale):
    rp, ci = csr(M)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    rpd, cid = torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV)
    o, lse, res = fa.forward_blocksparse(q, k, v, rpd, cid, causal=causal, scale=scale, residual=True)
    g = fa.backward_blocksparse(q, k, v, rpd, cid, o, lse, do, causal=causal, scale=scale, o_residual=res)
    torch.cuda.synchronize()
    return g, rp, ci


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,density", CASES)
def test_backward_random_tables(B, Hq, Hkv, Nq, Nk, d, causal, density):
    g = np.random.default_rng(Nq + Nk + d + 1)
    nqt, nkt = -(-Nq // 128), -(-Nk // 128)
    M = g.random((nqt, nkt)) < density
    M[np.arange(nqt), np.arange(nqt) % nkt] = True
    M[1] = False                                               # a query tile that sees nothing
    M[:, nkt - 2] = False                                      # a key tile no query tile lists
    x = inputs.shape_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq + d + 7)
    scale = 1 / np.sqrt(d)
    (dq, dk, dv), rp, ci = run_bwd(x, M, causal, scale)
    rq, rk, rv = A.attention_blocksparse_backward(x["q"], x["k"], x["v"], x["do"], rp, ci, scale, causal)
    tag = f"blocksparse bwd {B}x{Hq}/{Hkv} {Nq}x{Nk} d={d} causal={causal}"
    assert_grad(dq, rq, "dQ " + tag)
    assert_grad(dk, rk, "dK " + tag)
    assert_grad(dv, rv, "dV " + tag)
    assert not f64(dq[:, 128:256]).any()                          # the query tile that sees nothing
    dead = slice((nkt - 2) * 128, (nkt - 1) * 128)
    assert not f64(dk[:, dead]).any() and not f64(dv[:, dead]).any()


@pytest.mark.parametrize("causal,d", [(False, 128), (True, 64)])
def test_backward_every_tile_listed_equals_the_dense_kernels(causal, d):
    """Both backward calls take the block-sparse forward's O, LSE and residual (the
    dense forward without a mask may split keys and round O differently), so the
    two backward paths see the same inputs and must agree bit for bit."""
    N = 1000
    x = inputs.shape_inputs(1, 4, 2, N, N, d, seed=5)
    nt = -(-N // 128)
    rp, ci = csr(np.ones((nt, nt), bool))
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    rpd, cid = torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV)
    o, lse, res = fa.forward_blocksparse(q, k, v, rpd, cid, causal=causal, scale=0.1, residual=True)
    g1 = fa.backward_blocksparse(q, k, v, rpd, cid, o, lse, do, causal=causal, scale=0.1, o_residual=res)
    g2 = fa.backward(q, k, v, o, lse, do, causal=causal, scale=0.1, o_residual=res)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


# ------------------------------------------------------------------ split key tiles
def _ru(x, a=256):
    return -(-x // a) * a


def plan_rule(M, causal, B, Hkv, g):
    """The dK/dV segment rule, written out on the host: per key tile n = g x (query
    tiles listing it, tiles above the diagonal dropped under causal); seg =
    max(32, ceil(B Hkv sum(n) / 152)); a tile with n > seg becomes ceil(n / seg)
    segments, each with its own partial tile."""
    Mc = M & np.tril(np.ones_like(M)) if causal else M
    n = g * Mc.sum(axis=0)
    seg = max(32, -(-(B * Hkv * int(n.sum())) // 152))
    return seg, np.where(n > seg, -(-n // seg), 1)


def plan_header(ws, B, Hq, Nq, Nk, nnz):
    """[segments, partial slots, split tiles, seg] of the plan in a block-sparse
    backward workspace (after the status header, the -LSE2 and -D rows, the two
    list pointer arrays and the two index arrays)."""
    nqt, nkt = -(-Nq // 128), -(-Nk // 128)
    off = 256 + 2 * _ru(B * Hq * nqt * 128 * 4) + _ru((nqt + 1) * 4) + _ru((nkt + 1) * 4) + 2 * _ru(nnz * 4 + 4)
    return ws[off:off + 16].view(torch.int32).cpu().numpy()


SPLIT_CASES = [  # B, Hq, Hkv, N, d, causal, local tiles (+ key tile 0 for everyone; not causal: + the last)
    (1, 4, 1, 4096, 128, True, 3),
    (2, 8, 2, 2048, 64, False, 2),
    (1, 8, 2, 2000, 128, False, 2),   # the split last key tile is ragged (80 of 128 keys)
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,local", SPLIT_CASES)
def test_backward_split_key_tiles(B, Hq, Hkv, N, d, causal, local):
    """Key tiles every query tile lists have more iterations than a segment: the
    plan splits them, their fp32 partial tiles are summed in segment order.
    Checks the plan against the rule, the gradients against the oracle and that
    two calls agree bit for bit."""
    nt = -(-N // 128)
    M = np.array(inputs.local_global_tiles(nt, local, 1))
    if not causal:
        M[:, nt - 1] = True
    seg, nseg = plan_rule(M, causal, B, Hkv, Hq // Hkv)
    assert (nseg > 1).any()
    x = inputs.shape_inputs(B, Hq, Hkv, N, N, d, seed=N + d + 11)
    scale = 1 / np.sqrt(d)
    rp, ci = csr(M)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    rpd, cid = torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV)
    o, lse, res = fa.forward_blocksparse(q, k, v, rpd, cid, causal=causal, scale=scale, residual=True)
    s = fa.binding._dims(q, k, scale, causal)
    ws = torch.zeros(fa.library().fa_bwd_blocksparse_workspace_size(fa.binding.ctypes.byref(s), len(ci)),
                     dtype=torch.uint8, device=DEV)
    grads = []
    for _ in range(2):
        g = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        fa.fa_bwd_blocksparse(q, k, v, rpd, cid, o, lse, do, *g, s, ws, res)
        torch.cuda.synchronize()
        grads.append(g)
    rc, st = fa.binding.device_status(ws)
    assert rc == 0 and st == 0
    hdr = plan_header(ws, B, Hq, N, N, len(ci))
    assert list(hdr) == [int(nseg.sum()), int(nseg[nseg > 1].sum()), int((nseg > 1).sum()), seg]
    for a, b in zip(*grads):
        assert torch.equal(a, b)
    rq, rk, rv = A.attention_blocksparse_backward(x["q"], x["k"], x["v"], x["do"], rp, ci, scale, causal)
    tag = f"split blocksparse bwd {B}x{Hq}/{Hkv} N={N} d={d} causal={causal}"
    dq, dk, dv = grads[0]
    assert_grad(dq, rq, "dQ " + tag)
    assert_grad(dk, rk, "dK " + tag)
    assert_grad(dv, rv, "dV " + tag)


@pytest.mark.slow
def test_backward_local_global_n16384_sampled():
    """The block-sparse backward at the bench's workload (local 8 + global 1, causal,
    GQA 32/8, N = 16384, d = 128), where the global key tile is split: sampled rows
    of dQ and of one K/V head's dK, dV (the global tile's among them) against the
    oracle."""
    w = inputs.BLOCKSPARSE_N16384
    nt = w.Nq // 128
    M = np.array(inputs.local_global_tiles(nt, w.extra["local_tiles"], w.extra["global_tiles"]))
    seg, nseg = plan_rule(M, w.causal, w.B, w.Hkv, w.Hq // w.Hkv)
    assert nseg[0] > 1
    x = inputs.make(w, device=DEV)
    rp, ci = csr(M)
    rpd, cid = torch.from_numpy(rp).to(DEV), torch.from_numpy(ci).to(DEV)
    o, lse, res = fa.forward_blocksparse(x["q"], x["k"], x["v"], rpd, cid, causal=True, scale=w.scale, residual=True)
    dq, dk, dv = fa.backward_blocksparse(x["q"], x["k"], x["v"], rpd, cid, o, lse, x["do"], causal=True,
                                         scale=w.scale, o_residual=res)
    torch.cuda.synchronize()
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    rng = np.random.default_rng(23)
    b, kvh, g = 0, 5, w.Hq // w.Hkv
    q_rows = np.unique(np.concatenate([[0, 127, 77 * 128 + 3, w.Nq - 1], rng.integers(0, w.Nq, 12)]))
    k_rows = np.unique(np.concatenate([[0, 5, 127, 77 * 128 + 3, w.Nk - 1], rng.integers(0, w.Nk, 12)]))
    xc = {n: x[n].cpu() for n in ("q", "k", "v", "do")}
    sk = np.zeros((len(k_rows), w.d))
    sv = np.zeros((len(k_rows), w.d))
    for h in range(kvh * g, (kvh + 1) * g):
        rq, rk, rv = A.attention_blocksparse_backward_sampled(xc["q"], xc["k"], xc["v"], xc["do"], rp, ci, w.scale,
                                                              True, b, h, q_rows, k_rows)
        assert_grad(dq[b, q_rows, h], rq, f"dQ b{b} h{h}")
        sk += rk
        sv += rv
    assert_grad(dk[b, k_rows, kvh], sk, f"dK b{b} kvh{kvh}")
    assert_grad(dv[b, k_rows, kvh], sv, f"dV b{b} kvh{kvh}")
