"""GPU parity of the FP8 path against the oracle: the tensor-core building
blocks with E4M3 operands, the quantiser (codes bit-exact), and the FP8 forward."""

import numpy as np
import pytest
import torch

import exact_io_aware_21_gb300 as fa
from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from oracle import fp8 as F
from parity import assert_fwd, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRAD_BOUND_MIXED = 0.05  # twice the largest measured (0.025 on GB300)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.library().fa_set_wait_timeout_ns(10_000_000_000)


def status_ok(ws):
    rc, st = fa.binding.device_status(ws)
    assert rc == 0 and st == 0, f"device status {st:#x}"


def codes(shape, seed, max_exp=12):
    """Random finite E4M3 codes with exponent field at most max_exp."""
    g = np.random.default_rng(seed)
    c = g.integers(0, 256, shape).astype(np.uint8)
    e = (c >> 3) & 15
    c = np.where(e > max_exp, (c & 0x87) | (max_exp << 3), c).astype(np.uint8)
    return c


# ------------------------------------------------------------------ building blocks
def run_selftest(mode, a, b):
    c = torch.zeros(128, 128, dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    da, db = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    fa.binding.check(fa.library().fa_selftest_mma(mode, 128, da.data_ptr(), db.data_ptr(), c.data_ptr(),
                                                  ws.data_ptr(), None))
    torch.cuda.synchronize()
    status_ok(ws)
    return c.cpu().double().numpy()


def test_selftest_e4m3_qk_form():
    a, b = codes((128, 128), 1), codes((128, 128), 2)
    ref = F.e4m3_decode(a) @ F.e4m3_decode(b).T
    np.testing.assert_allclose(run_selftest(2, a, b), ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())


def test_selftest_e4m3_pv_form():
    a, b = codes((128, 128), 3), codes((128, 128), 4)
    ref = F.e4m3_decode(a) @ F.e4m3_decode(b)
    np.testing.assert_allclose(run_selftest(3, a, b), ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())


# ------------------------------------------------------------------ quantiser

def signs_for(d, use):
    return inputs.hadamard_signs(d, seed=d).to(DEV) if use else None


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("block_rows", [128, 0])
@pytest.mark.parametrize("had", [False, True])
def test_quantize_codes_and_scales_bit_exact(d, block_rows, had):
    B, N, H = 2, 300, 3                                        # three row blocks, the last ragged
    x = inputs.shape_inputs(B, H, H, N, N, d, seed=7 + d, with_do=False)["q"]
    x = x * torch.tensor([0.01, 1.0, 30.0]).view(1, 1, H, 1).to(torch.bfloat16)   # one scale range per head
    x[1, 128:256, 0] = 0                                       # an all-zero block
    sg = signs_for(d, had)
    codes, sc = fa.quantize_fp8(x.to(DEV), block_rows, sg)
    torch.cuda.synchronize()
    ref_codes, ref_sc = F.quantize(x.float().numpy(), block_rows, None if sg is None else sg.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert np.array_equal(sc.cpu().numpy(), ref_sc)


def test_quantize_strided_views():
    x = inputs.shape_inputs(1, 4, 4, 256, 256, 128, seed=3, with_do=False)["q"].to(DEV)
    xv = x[:, :, 1:3]                                          # a head slice: strided rows
    out = torch.zeros((1, 256, 4, 128), dtype=torch.uint8, device=DEV)[:, :, 1:3]
    sc = torch.full((1, 2, 2), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(fa.library().fa_quantize_fp8_workspace_size(1, 2), dtype=torch.uint8, device=DEV)
    fa.fa_quantize_fp8(xv, 128, None, out, sc, ws)
    torch.cuda.synchronize()
    ref_codes, ref_sc = F.quantize(xv.cpu().float().numpy(), 128)
    assert np.array_equal(out.cpu().numpy(), ref_codes) and np.array_equal(sc.cpu().numpy(), ref_sc)


# ------------------------------------------------------------------ forward
def fp8_inputs(B, Hq, Hkv, N, seed, had, outliers=False, causal=False):
    w = inputs.Workload("t", B, Hq, Hkv, N, N, 128, causal, outliers=outliers, seed=seed)
    x = inputs.make(w, with_do=True)
    sg = signs_for(128, had)
    q8, sq = fa.quantize_fp8(x["q"].to(DEV), 128, sg)
    k8, sk = fa.quantize_fp8(x["k"].to(DEV), 128, sg)
    v8, sv = fa.quantize_fp8(x["v"].to(DEV), 0, None)
    return x, (q8, k8, v8, sq, sk, sv)


def cpu(t):
    return t.cpu().numpy()


CASES = [  # B, Hq, Hkv, N, causal, window, Hadamard
    (1, 2, 1, 300, False, None, False),
    (2, 4, 2, 512, True, None, False),
    (1, 4, 4, 384, False, (100, 20), True),
    (1, 8, 2, 1024, True, None, True),
    (1, 2, 2, 200, True, (64, 0), False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,causal,window,had", CASES)
def test_forward_fp8_matches_oracle(B, Hq, Hkv, N, causal, window, had):
    x, (q8, k8, v8, sq, sk, sv) = fp8_inputs(B, Hq, Hkv, N, seed=N + Hq, had=had)
    scale = 1 / np.sqrt(128)
    o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    o_ref, lse_ref = F.attention_forward_fp8(cpu(q8), cpu(k8), cpu(v8), cpu(sq), cpu(sk), cpu(sv), scale, causal,
                                             window)
    tag = f"fp8 {B}x{Hq}/{Hkv}x{N} causal={causal} window={window} hadamard={had}"
    assert_fwd(o, lse, o_ref, lse_ref, tag)
    # and the whole FP8 scheme against exact attention on these N(0,1) inputs
    o_ex, _ = A.attention_forward(x["q"], x["k"], x["v"], scale, causal, window=window)
    assert rel_fro(o, o_ex) < 0.08, tag


def test_forward_fp8_zero_blocks():
    """An all-zero Q block and an all-zero K block (scale 0): S = 0 there, no NaN."""
    B, H, N = 1, 2, 384
    x = inputs.shape_inputs(B, H, H, N, N, 128, seed=5, with_do=False)
    x["q"][0, 128:256, 0] = 0
    x["k"][0, 256:384, 1] = 0
    q8, sq = fa.quantize_fp8(x["q"].to(DEV), 128)
    k8, sk = fa.quantize_fp8(x["k"].to(DEV), 128)
    v8, sv = fa.quantize_fp8(x["v"].to(DEV), 0)
    for causal in (False, True):
        o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
        torch.cuda.synchronize()
        o_ref, lse_ref = F.attention_forward_fp8(cpu(q8), cpu(k8), cpu(v8), cpu(sq), cpu(sk), cpu(sv),
                                                 1 / np.sqrt(128), causal)
        assert_fwd(o, lse, o_ref, lse_ref, f"zero blocks causal={causal}")


@pytest.mark.slow
def test_forward_fp8_full_size_sampled():
    """The benchmark's FP8 leg: GQA causal N = 8192 with the outlier channel,
    Hadamard rotation on; oracle on sampled query blocks of a few heads."""
    w = inputs.GQA_N8192_D128
    x = inputs.make(w, device=DEV, with_do=False)
    sg = signs_for(128, True)
    q8, sq = fa.quantize_fp8(x["q"], 128, sg)
    k8, sk = fa.quantize_fp8(x["k"], 128, sg)
    v8, sv = fa.quantize_fp8(x["v"], 0, None)
    o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    heads = [(0, 0), (0, 13), (0, 31)]
    blocks = [0, 31, 63]
    o_ref, lse_ref = F.attention_forward_fp8(cpu(q8), cpu(k8), cpu(v8), cpu(sq), cpu(sk), cpu(sv), w.scale, True,
                                             heads=heads, q_blocks=blocks)
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    for b, h in heads:
        assert_fwd(o[b, rows, h], lse[b, h, rows], o_ref[b, rows, h], lse_ref[b, h, rows], f"fp8 full h{h}")
    # the whole FP8 scheme against exact attention on these outlier inputs: the same
    # relative bound as the small cases (the pages' MSE level is for N(0,1) data, below)
    o_ex, _ = A.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), w.scale, True, heads=heads, rows=rows)
    for b, h in heads:
        assert rel_fro(o[b, rows, h], o_ex[b, rows, h]) < 0.08, f"fp8 vs exact attention h{h}"


@pytest.mark.slow
@pytest.mark.parametrize("had", [False, True])
def test_forward_fp8_error_at_the_pages_level(had):
    """The pages' error level for the whole FP8 scheme ("第18章" §18.6.2, Table 18-21:
    d = 128, N = 8192, MSE below 5e-5 against exact attention), checked on the GPU
    output itself: the GQA causal N = 8192 shape with N(0, 1) inputs, sampled query
    blocks of a few heads, with and without the Hadamard rotation."""
    w = inputs.Workload("fp8_table", 1, 32, 8, 8192, 8192, 128, True, seed=9)
    x, (q8, k8, v8, sq, sk, sv) = fp8_inputs(w.B, w.Hq, w.Hkv, w.Nq, seed=9, had=had, causal=True)
    o, _ = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    heads = [(0, 0), (0, 17), (0, 31)]
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in (0, 20, 63)])
    o_ex, _ = A.attention_forward(x["q"], x["k"], x["v"], w.scale, True, heads=heads, rows=rows)
    for b, h in heads:
        mse = float(np.mean((o[b, rows, h].float().cpu().numpy() - o_ex[b, rows, h]) ** 2))
        assert mse < 5e-5, f"fp8 vs exact attention h{h} hadamard={had}: MSE {mse:.2e}"


@pytest.mark.parametrize("had", [True, False])
def test_fp8_forward_then_bf16_backward(had):
    """The pages' mixed mode ("第18章" §18.6.2, after Table 18-21): the forward in FP8,
    the backward in bf16.  The bf16 backward takes the FP8 forward's O and LSE with the
    bf16 Q, K, V, so P rebuilt from bf16 scores carries the FP8 forward's LSE error.
    On N(0, 1) inputs every gradient stays within a relative Frobenius distance of
    0.05 of the exact gradients (fp64 oracle), the FP8 output within 0.08.  (With the
    outlier channel the FP8 LSE is off by whole units for peaky rows and P rebuilt
    from exact scores no longer sums to one there: dQ was 2.8x off in relative
    Frobenius distance.  The mixed mode needs statistics consistent with the
    backward's own scores, which the FP8 forward does not give on such data.)"""
    outliers = False
    B_, Hq, Hkv, N = 1, 4, 2, 768
    x, (q8, k8, v8, sq, sk, sv) = fp8_inputs(B_, Hq, Hkv, N, seed=77, had=had, outliers=outliers, causal=True)
    scale = 1 / np.sqrt(128)
    o, lse = fa.forward_fp8(q8, k8, v8, sq, sk, sv, causal=True, scale=scale)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    o_ex, _ = A.attention_forward(x["q"], x["k"], x["v"], scale, True)
    dq_ex, dk_ex, dv_ex = A.attention_backward(x["q"], x["k"], x["v"], x["do"], scale, True)
    errs = {"O": rel_fro(o, o_ex), "dQ": rel_fro(dq, dq_ex), "dK": rel_fro(dk, dk_ex), "dV": rel_fro(dv, dv_ex)}
    print("fp8 forward + bf16 backward, hadamard", had, "outliers", outliers, {n: f"{e:.3g}" for n, e in errs.items()})
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    assert errs["O"] < 0.08
    for n in ("dQ", "dK", "dV"):
        assert errs[n] < GRAD_BOUND_MIXED, (n, errs)
