"""FP8 (E4M3) attention forward with per-block scales and incoherent processing.

TEST INFRASTRUCTURE ONLY (see the package docstring).  numpy; the quantiser's
rounding decisions are taken in float32 (the kernel's precision, where the
pages fix none), everything else in float64.

Definitions followed (one bullet per function below):
  * E4M3 ("第18章 FlashAttention" §18.6.2 and Fig. 18-24): 1 sign bit, 4
    exponent bits (bias 7), 3 mantissa bits; no infinities, NaN = exponent and
    mantissa all ones, so the largest finite magnitude is 1.75 * 2^8 = 448 and
    the smallest subnormal 2^-9.  Encoding rounds to nearest with ties to even
    and saturates magnitudes above 448 to 448 (the quantiser never exceeds 448
    by more than a rounding error, so saturation only absorbs that error).
  * fast Walsh-Hadamard transform: the radix-2 butterflies (a, b) -> (a + b,
    a - b) at strides 1, 2, 4, ..., d/2, i.e. multiplication by the Sylvester
    Hadamard matrix H_d (symmetric, H_d H_d = d I).
  * incoherent processing ("CMU 11-868 L21" notes, slide 24): Q and K are both
    multiplied by one random orthogonal matrix J, which leaves Q K^T unchanged
    ((QJ)(KJ)^T = Q K^T) and spreads outlier channels over all channels.  J =
    diag(sigma) H_d / sqrt(d) with sigma a vector of random signs (passed in).
  * per-block quantisation (§18.6.2, part 2): X_fp8 = quant_E4M3(X / s) with
    s = max|X| / 448, one scale per loaded block of Q and of K (128 rows of
    one head, the kernel's tile); V, for which the pages give no block rule,
    takes one scale per (batch, head).
  * FP8 forward: the FlashAttention-2 loop (§18.5: per query block, key blocks
    in order, running row max, unnormalised output, O / l at the end) with S
    formed from the E4M3 operands and their scales, the softmax in full
    precision, and P passed to the P V product as E4M3 with the scale its
    bound fixes: P <= 1, so s_P = 1 / 448 and the product reads 448 P.
"""

import numpy as np

from .attention import causal_mask, window_mask

E4M3_MAX = 448.0
P_SCALE = 448.0          # P is quantised as 448 * P (s_P = 1 / 448)
LOG2E = 1.4426950408889634


# ----------------------------------------------------------------------------- E4M3
def e4m3_encode(x):
    """Round each value to E4M3 (nearest, ties to even, saturating at 448).

    ``x`` is any float array; its values are taken exactly (as float64) and
    rounded once.  Returns uint8 codes.  NaN inputs are not expected."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << 7
    a = np.minimum(np.abs(x), E4M3_MAX)
    code = np.zeros(a.shape, dtype=np.int64)
    nz = a > 0
    _, E = np.frexp(np.where(nz, a, 1.0))        # a = f * 2^E, f in [0.5, 1)
    e = E - 1                                    # a in [2^e, 2^(e+1))
    normal = nz & (e >= -6)
    # normal: 3 fraction bits -> a / 2^(e-3) in [8, 16), rounded half to even
    q = np.rint(np.where(normal, np.ldexp(a, -(e - 3)), 0.0)).astype(np.int64)
    carry = q == 16                              # rounding reached the next binade
    e_n = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    code = np.where(normal, ((e_n + 7) << 3) | (q - 8), code)
    # subnormal: a / 2^-9 in [0, 8), rounded half to even (8 is the smallest normal)
    sub = nz & ~normal
    qs = np.rint(np.where(sub, np.ldexp(a, 9), 0.0)).astype(np.int64)
    code = np.where(sub, qs, code)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(codes):
    """Value of each E4M3 code as float64 (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


# ----------------------------------------------------------------------------- Hadamard
def fwht(x):
    """Unnormalised fast Walsh-Hadamard transform along the last axis, in x's dtype.

    Butterflies at strides h = 1, 2, ..., d/2: the element pair (j, j + h) of
    every 2h-block becomes (sum, difference)."""
    x = np.array(x, copy=True)
    d = x.shape[-1]
    if d & (d - 1):
        raise ValueError("the transform needs a power-of-two length")
    lead = x.shape[:-1]
    h = 1
    while h < d:
        y = x.reshape(lead + (d // (2 * h), 2, h))
        a, b = y[..., 0, :], y[..., 1, :]
        x = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        h *= 2
    return x


def incoherent(x, signs):
    """x J with J = diag(signs) H_d / sqrt(d), in float64."""
    x = np.asarray(x, dtype=np.float64) * np.asarray(signs, dtype=np.float64)
    return fwht(x) / np.sqrt(x.shape[-1])


# ----------------------------------------------------------------------------- quantiser
def quantize(x, block_rows=128, signs=None):
    """E4M3 codes and scales of x [B, N, H, d] (values taken as float32).

    ``block_rows`` > 0: one scale per block of that many rows of one head,
    scales [B, H, ceil(N / block_rows)]; 0: one scale per (batch, head),
    scales [B, H].  With ``signs`` the rows are first transformed by J
    (incoherent processing).  Arithmetic, in float32 like the kernel: y =
    fwht(signs * x) (unnormalised), amax = max|y| over the block, inv = 448 /
    amax, code = E4M3(y * inv), scale = amax / 448, times 1 / sqrt(d) when
    transformed (so that code * scale approximates x J).  An all-zero block
    gets codes 0 and scale 0.
    """
    y = np.asarray(x, dtype=np.float32)
    B, N, H, d = y.shape
    if signs is not None:
        y = fwht(y * np.asarray(signs, dtype=np.float32))
    rows = block_rows if block_rows > 0 else N
    nblk = -(-N // rows)
    codes = np.zeros(y.shape, dtype=np.uint8)
    scales = np.zeros((B, H, nblk), dtype=np.float32)
    four48 = np.float32(E4M3_MAX)
    for b in range(B):
        for h in range(H):
            for k in range(nblk):
                blk = y[b, k * rows:(k + 1) * rows, h, :]
                amax = np.float32(np.max(np.abs(blk)))
                if amax == 0:
                    continue
                inv = np.float32(four48 / amax)
                codes[b, k * rows:(k + 1) * rows, h, :] = e4m3_encode(np.float32(blk * inv))
                s = np.float32(amax / four48)
                if signs is not None:
                    s = np.float32(s * np.float32(1.0 / np.sqrt(d)))
                scales[b, h, k] = s
    return codes, (scales if block_rows > 0 else scales[:, :, 0])


def dequantize(codes, scales, block_rows=128):
    """codes * scale as float64 [B, N, H, d] (the inverse map of ``quantize``)."""
    vals = e4m3_decode(codes)
    B, N, H, d = vals.shape
    sc = np.asarray(scales, dtype=np.float64)
    if block_rows > 0:
        per_row = np.repeat(sc, block_rows, axis=2)[:, :, :N]      # [B, H, N]
    else:
        per_row = np.repeat(sc[:, :, None], N, axis=2)
    return vals * per_row.transpose(0, 2, 1)[..., None]


# ----------------------------------------------------------------------------- forward
def attention_forward_fp8(q8, k8, v8, sq, sk, sv, scale, causal=False, window=None, block=128,
                          quantize_p=True, heads=None, q_blocks=None):
    """FP8 forward: O [B, Nq, Hq, d] and LSE [B, Hq, Nq] (natural log), float64.

    q8, k8, v8: E4M3 codes; sq [B, Hq, ceil(Nq/block)], sk [B, Hkv, ceil(Nk/block)]
    per-block scales, sv [B, Hkv] per-head scales.  Query head h reads KV head
    h // (Hq // Hkv).  Per query block of ``block`` rows, key blocks of
    ``block`` keys in ascending order (those no row of the block can see are
    skipped; they would contribute nothing):
        x = (Q K_j^T) * scale * log2(e)      (base-2 logits from the dequantised operands)
        m_new = max(m, rowmax x);  alpha = 2^(m - m_new)
        P' = 448 * 2^(x - m_new);  l = alpha l + rowsum P'
        O = alpha O + E4M3(P') V_j           (V as codes; its scale applied at the end)
    then O * sv / l and LSE = (m + log2 l - log2 448) ln 2.  ``quantize_p``
    False keeps P' unrounded (the loop alone, for pinning).  ``heads`` (list of
    (b, h)) and ``q_blocks`` (query block indices) restrict what is computed;
    the rest stays NaN.
    """
    Qd = dequantize(q8, sq, block)
    Kd = dequantize(k8, sk, block)
    Vc = e4m3_decode(v8)
    B, Nq, Hq, d = Qd.shape
    Nk, Hkv = Kd.shape[1], Kd.shape[2]
    if (causal or window is not None) and Nq != Nk:
        raise ValueError("causal and windowed attention are defined here for Nq == Nk only")
    g = Hq // Hkv
    o = np.full((B, Nq, Hq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    c = scale * LOG2E
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]):
        kv = h // g
        for i0 in (range(0, Nq, block) if q_blocks is None else [qb * block for qb in q_blocks]):
            rows = np.arange(i0, min(Nq, i0 + block))
            m = np.full(len(rows), -np.inf)
            l = np.zeros(len(rows))
            O = np.zeros((len(rows), d))
            for j0 in range(0, Nk, block):
                cols = np.arange(j0, min(Nk, j0 + block))
                x = (Qd[b, rows, h, :] @ Kd[b, cols, kv, :].T) * c
                hidden = np.zeros(x.shape, dtype=bool)
                if causal:
                    hidden |= causal_mask(rows, Nk)[:, cols]
                if window is not None:
                    hidden |= window_mask(rows, Nk, *window)[:, cols]
                if hidden.all():
                    continue
                x = np.where(hidden, -np.inf, x)
                m_new = np.maximum(m, x.max(axis=1))
                ref = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp2(m - ref), 0.0)
                Pp = P_SCALE * np.exp2(x - ref[:, None])
                l = alpha * l + Pp.sum(axis=1)
                P8 = e4m3_decode(e4m3_encode(Pp)) if quantize_p else Pp
                O = alpha[:, None] * O + P8 @ Vc[b, cols, kv, :]
                m = m_new
            o[b, rows, h, :] = O * float(sv[b, kv]) / l[:, None]
            lse[b, h, rows] = (m + np.log2(l) - np.log2(P_SCALE)) * np.log(2.0)
    return o, lse
