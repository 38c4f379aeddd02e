"""Pins of the FP8 oracle (no GPU): the E4M3 codec, the Hadamard transform, the
per-block quantiser, and the FP8 forward loop.

Against: torch's float8_e4m3fn conversions (a library routine for the same
format), scipy's Sylvester Hadamard matrix, hand-computed codes, the plain
attention definition on exactly representable operands, the E4M3 rounding
bound for P, the pages' printed error levels (Table 18-21) and the pages'
claim that the random Hadamard rotation lowers the quantisation error on
outlier data (lecture slide 24).
"""

import numpy as np
import pytest
import torch

from exact_io_aware_21_gb300 import inputs
from oracle import attention as A
from oracle import fp8 as F

RNG = np.random.default_rng(11)


# ----------------------------------------------------------------------------- E4M3
def test_decode_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    mine = F.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    assert np.array_equal(mine[~np.isnan(mine)], lib[~np.isnan(lib)])
    assert np.nanmax(mine) == 448.0 and np.nanmin(np.abs(mine[mine != 0])) == 2.0 ** -9
    assert set(np.flatnonzero(np.isnan(mine))) == {0x7F, 0xFF}


def test_encode_matches_library_including_ties():
    vals = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = np.sort(vals[np.isfinite(vals)])
    mids = (finite[:-1] + finite[1:]) / 2                      # every rounding tie
    x = np.concatenate([RNG.standard_normal(50000) * 30, RNG.standard_normal(50000) * 1e-3,
                        RNG.uniform(-448, 448, 50000), finite, mids]).astype(np.float32)
    x = np.clip(x, -448, 448)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), lib)


@pytest.mark.parametrize("x,code", [(448.0, 0x7E), (500.0, 0x7E), (-1e6, 0xFE), (2.0 ** -9, 0x01),
                                    (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (1.0625, 0x38),
                                    (1.1875, 0x3A), (-0.0, 0x80), (0.0, 0x00), (240.0, 0x77),
                                    (2.0 ** -6, 0x08), (0.875 * 2.0 ** -6, 0x07)])
def test_encode_known_values(x, code):
    # ties go to the even mantissa (1.0625 -> 1.0, 1.1875 -> 1.25, 1.5*2^-9 -> 2*2^-9);
    # above 448 saturates; 2^-6 is the smallest normal, 7*2^-9 the largest subnormal
    assert int(F.e4m3_encode(np.array([x]))[0]) == code


# ----------------------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_fwht_is_the_sylvester_hadamard_matrix(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(d).astype(np.float64)
    x = RNG.standard_normal((5, d))
    assert np.allclose(F.fwht(x), x @ H.T, rtol=0, atol=1e-12)
    xi = RNG.integers(-50, 50, (4, d)).astype(np.float64)
    assert np.array_equal(F.fwht(F.fwht(xi)), d * xi)          # H H = d I, exactly on integers


def test_incoherent_processing_preserves_qk():
    d = 128
    s = inputs.hadamard_signs(d, seed=5).numpy()
    assert set(np.unique(s)) == {-1.0, 1.0}
    q, k = RNG.standard_normal((40, d)), RNG.standard_normal((30, d))
    J = F.incoherent(np.eye(d), s)
    assert np.allclose(J @ J.T, np.eye(d), atol=1e-13)
    assert np.allclose(F.incoherent(q, s) @ F.incoherent(k, s).T, q @ k.T, atol=1e-11)
    assert np.allclose(F.incoherent(q, s), q @ J, atol=1e-13)


# ----------------------------------------------------------------------------- quantiser
def test_quantize_hand_example():
    # amax 3.5: inv = 448 / 3.5 = 128 exactly; 0.5 -> 64, 1 -> 128, -3.5 -> -448
    x = np.zeros((1, 2, 1, 4), dtype=np.float32)
    x[0, 0, 0, :3] = [0.5, 1.0, -3.5]
    codes, sc = F.quantize(x, block_rows=128)
    assert list(codes[0, 0, 0]) == [0x68, 0x70, 0xFE, 0x00] and list(codes[0, 1, 0]) == [0, 0, 0, 0]
    assert sc.shape == (1, 1, 1) and sc[0, 0, 0] == np.float32(3.5 / 448)


@pytest.mark.parametrize("signs", [False, True])
@pytest.mark.parametrize("block_rows", [128, 0])
def test_quantize_bounds(signs, block_rows):
    d, N = 64, 300                                             # three blocks, the last ragged
    x = (RNG.standard_normal((2, N, 3, d)) * RNG.uniform(0.1, 10, (2, 1, 3, 1))).astype(np.float32)
    sg = inputs.hadamard_signs(d, seed=1).numpy() if signs else None
    codes, sc = F.quantize(x, block_rows, sg)
    target = F.incoherent(x, sg) if signs else x.astype(np.float64)
    deq = F.dequantize(codes, sc, block_rows)
    vals = F.e4m3_decode(codes)
    assert np.all(np.isfinite(vals)) and np.abs(vals).max() == 448.0
    rows = block_rows if block_rows else N
    for b in range(2):
        for h in range(3):
            for k0 in range(0, N, rows):
                blk = vals[b, k0:k0 + rows, h]
                assert np.abs(blk).max() == 448.0               # the block's largest element maps to 448
                s = sc[b, h, k0 // rows] if block_rows else sc[b, h]
                t, dq = target[b, k0:k0 + rows, h], deq[b, k0:k0 + rows, h]
                # half an E4M3 step: 2^-4 relative for normals, 2^-10 * s below 2^-6 * s,
                # plus float32 rounding of the transform and of the scale
                bound = np.maximum(2.0 ** -4 * np.abs(t), 2.0 ** -10 * s) * (1 + 1e-5) + 1e-6 * np.abs(t).max()
                assert np.all(np.abs(dq - t) <= bound)


def test_quantize_zero_block():
    x = np.zeros((1, 256, 1, 8), dtype=np.float32)
    x[0, 200, 0, 3] = 2.0
    codes, sc = F.quantize(x, 128)
    assert not codes[0, :128].any() and sc[0, 0, 0] == 0.0
    assert codes[0, 200, 0, 3] == 0x7E and sc[0, 0, 1] == np.float32(2.0 / 448)


# ----------------------------------------------------------------------------- forward
def random_codes(shape, rng):
    """E4M3 codes of finite values spread over the format's range."""
    c = rng.integers(0, 256, shape).astype(np.uint8)
    return np.where((c & 0x7F) == 0x7F, c & 0xF0, c).astype(np.uint8)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,window", [(1, 2, 1, 300, 64, False, None), (2, 2, 2, 257, 32, True, None),
                                                        (1, 4, 2, 384, 16, False, (100, 20)),
                                                        (1, 1, 1, 200, 16, True, (50, 0))])
def test_loop_without_p_rounding_is_plain_attention(B, Hq, Hkv, N, d, causal, window):
    rng = np.random.default_rng(N)
    nb = -(-N // 128)
    q8, k8, v8 = random_codes((B, N, Hq, d), rng), random_codes((B, N, Hkv, d), rng), random_codes((B, N, Hkv, d), rng)
    sq = np.ldexp(1.0, rng.integers(-9, -5, (B, Hq, nb))).astype(np.float32)
    sk = np.ldexp(1.0, rng.integers(-9, -5, (B, Hkv, nb))).astype(np.float32)
    sv = rng.uniform(0.001, 0.01, (B, Hkv)).astype(np.float32)
    scale = 0.3
    o8, l8 = F.attention_forward_fp8(q8, k8, v8, sq, sk, sv, scale, causal, window, quantize_p=False)
    q, k = F.dequantize(q8, sq), F.dequantize(k8, sk)
    v = F.e4m3_decode(v8) * sv[:, None, :, None].astype(np.float64)
    o, lse = A.attention_forward(q, k, v, scale, causal, window=window)
    assert np.allclose(o8, o, rtol=1e-11, atol=1e-13) and np.allclose(l8, lse, rtol=0, atol=1e-11)


def test_p_rounding_is_e4m3_at_scale_448():
    """Rounding P' = 448 P to E4M3 moves each output by at most half a step per term."""
    rng = np.random.default_rng(3)
    N, d = 256, 32
    q8, k8, v8 = random_codes((1, N, 1, d), rng), random_codes((1, N, 1, d), rng), random_codes((1, N, 1, d), rng)
    # scores of a few units, so that P spans E4M3's normal and subnormal ranges
    sq = np.full((1, 1, 2), 2.0 ** -11, np.float32)
    sk = np.full((1, 1, 2), 2.0 ** -11, np.float32)
    sv = np.ones((1, 1), np.float32)
    oq, lq = F.attention_forward_fp8(q8, k8, v8, sq, sk, sv, 1.0, quantize_p=True)
    o, l = F.attention_forward_fp8(q8, k8, v8, sq, sk, sv, 1.0, quantize_p=False)
    assert np.array_equal(lq, l)                            # l and m come from the unrounded P
    qd, kd, vd = F.dequantize(q8, sq)[0, :, 0], F.dequantize(k8, sk)[0, :, 0], F.e4m3_decode(v8)[0, :, 0]
    x = qd @ kd.T
    # relative to the final row max, each rounded P' (taken against the running max,
    # then scaled down by alpha <= 1) is off by at most 2^-4 P' or 2^-10
    Pp = 448.0 * np.exp(x - x.max(axis=1, keepdims=True))
    bound = ((2.0 ** -4 * Pp + 2.0 ** -10) @ np.abs(vd)) / Pp.sum(axis=1, keepdims=True)
    err = np.abs(oq - o)[0, :, 0]
    assert np.all(err <= bound * (1 + 1e-9)) and err.max() > 0


def test_p_reaches_the_product_as_e4m3_on_the_448_scale():
    """One key tile and V = I: O l' (l' = sum of 448 P, known here in closed form)
    recovers the P operand, which must be the E4M3 value nearest 448 P."""
    rng = np.random.default_rng(5)
    N = d = 128
    q8, k8 = random_codes((1, N, 1, d), rng), random_codes((1, N, 1, d), rng)
    sq = np.full((1, 1, 1), 2.0 ** -11, np.float32)
    sk = np.full((1, 1, 1), 2.0 ** -11, np.float32)
    v8 = np.where(np.eye(N, dtype=bool), 0x38, 0).astype(np.uint8)[None, :, None, :]   # 0x38 = 1.0
    scale = 100.0                                   # scores spread over E4M3's normal and subnormal ranges
    o, _ = F.attention_forward_fp8(q8, k8, v8, sq, sk, np.ones((1, 1), np.float32), scale)
    x = scale * (F.dequantize(q8, sq)[0, :, 0] @ F.dequantize(k8, sk)[0, :, 0].T)
    Pp = 448.0 * np.exp(x - x.max(axis=1, keepdims=True))
    P_op = o[0, :, 0] * Pp.sum(axis=1, keepdims=True)
    assert np.allclose(P_op, F.e4m3_decode(F.e4m3_encode(P_op)), rtol=1e-12, atol=0)   # on the E4M3 grid
    step = np.where(Pp >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(Pp, 1e-300))) - 3), 2.0 ** -9)
    assert np.all(np.abs(P_op - Pp) <= step / 2 * (1 + 1e-9))                        # the nearest one
    assert (Pp < 2.0 ** -6).mean() > 0.1 and (Pp > 1).mean() > 0.1                  # both ranges exercised


@pytest.mark.parametrize("d,N,mse_max", [(64, 4096, 1e-4), (128, 8192, 5e-5)])
def test_error_within_the_pages_table(d, N, mse_max):
    """Table 18-21: FP8 attention MSE below 1e-4 (d = 64, N = 4096) and 5e-5 (d = 128, N = 8192)."""
    w = inputs.Workload("t", 1, 1, 1, N, N, d, False, seed=3)
    x = inputs.make(w, with_do=False)
    q, k, v = (x[n].float().numpy() for n in ("q", "k", "v"))
    q8, sq = F.quantize(q, 128)
    k8, sk = F.quantize(k, 128)
    v8, sv = F.quantize(v, 0)
    blocks = [0, N // 128 - 1]
    o8, _ = F.attention_forward_fp8(q8, k8, v8, sq, sk, sv, w.scale, q_blocks=blocks)
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    o, _ = A.attention_forward(q, k, v, w.scale, rows=rows)
    mse = np.mean((o8[0, rows, 0] - o[0, rows, 0]) ** 2)
    assert mse < mse_max
    assert np.linalg.norm(o8[0, rows, 0] - o[0, rows, 0]) / np.linalg.norm(o[0, rows, 0]) < 0.08


@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_lowers_qk_quantisation_error_on_outliers(d):
    """Lecture slide 24: the random Hadamard rotation lowers the quantisation error on
    data with outliers (by 2.6x in the slide's simulation); without outliers it
    changes little."""
    signs = inputs.hadamard_signs(d, seed=2).numpy()

    def rel_err(x, sg):
        q, k = (x[n].float().numpy() for n in ("q", "k"))
        S = np.einsum("bnhd,bmhd->bhnm", q.astype(np.float64), k.astype(np.float64))
        q8, sq = F.quantize(q, 128, sg)
        k8, sk = F.quantize(k, 128, sg)
        Sq = np.einsum("bnhd,bmhd->bhnm", F.dequantize(q8, sq), F.dequantize(k8, sk))
        return np.linalg.norm(Sq - S) / np.linalg.norm(S)

    out = inputs.make(inputs.Workload("o", 1, 2, 2, 512, 512, d, False, outliers=True, seed=4), with_do=False)
    assert rel_err(out, None) > 2.6 * rel_err(out, signs)
    plain = inputs.make(inputs.Workload("p", 1, 2, 2, 512, 512, d, False, seed=4), with_do=False)
    assert 0.9 < rel_err(plain, None) / rel_err(plain, signs) < 1.1
