"""fp64 CPU oracle: scaled-dot-product attention, its gradients, and FlashDecoding.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64.

Tensor layout everywhere: ``[B, N, H, d]`` (batch, sequence, head, head dim), as
in the ``flash_attn_func`` interface of "第18章 FlashAttention" §18.7.1.  K and V
carry ``Hkv`` heads; query head ``h`` reads KV head ``h // (Hq // Hkv)``
(consecutive grouping; §18.2.2 says groups of query heads share one K/V head but
not which ones, so the plainest grouping is taken).  LSE is ``[B, Hq, Nq]``.

Definitions followed (one bullet per function below):
  * forward: S = scale * Q K^T, causal S_ij = -inf for j > i, P = softmax(S)
    row-wise with the max subtracted first (safe softmax), O = P V,
    LSE_i = m_i + ln(sum_j exp(S_ij - m_i)).  "第18章" §18.1.1 code listing and
    §18.2.1 (score, scaling, softmax), §18.2.2 (causal mask), §18.4.2 (safe
    softmax), Fig. 18-6 (the saved statistic is the log-sum-exp).
  * backward: dV = P^T dO, dP = dO V^T, D = rowsum(P * dP), dS = P * (dP - D),
    dQ = scale dS K, dK = scale dS^T Q; for grouped heads dK/dV sum over the
    group (chain rule through the broadcast).  §18.2.4 and §18.4.4 gradient
    formulas; D is taken over the whole row, as its definition states.
  * tiled forward: the outer/inner loop with running max m and sum l of
    §18.4.1 and the online update of §18.4.2; CMU 11-868 L21 notes slide 12
    (two-block rescaling) and its Algorithm-1 remark.
  * conditional rescaling (the L21 notes on FA4: an online-softmax variant
    that skips most rescalings): the same loop with a reference that moves
    only when a block's max passes it by more than a threshold.
  * FlashDecoding: each KV split t yields (m_t, l_t, O_t) with O_t the
    unnormalised local output; the combine is O = sum_t O_t e^{m_t - m} /
    sum_t l_t e^{m_t - m}.  §18.8.2 and lecture slides 57-60.
  * sliding window: query i sees keys j with i - left <= j <= i + right
    (``window_size=(left, right)`` of flash_attn_func, §18.7.1; local attention,
    §18.8.1), a negative bound meaning unbounded; with causal, j <= i as well.
    Like causal it is defined here for Nq == Nk (top-left aligned).
  * packed variable-length sequences (``flash_attn_varlen_func``, §18.7.1):
    Q [total_q, Hq, d] and K, V [total_k, Hkv, d] hold the sequences one after
    another; sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 and attends
    only within itself (no attention across sequence boundaries; causal is
    applied with the sequence's own positions).  LSE is [Hq, total_q].
  * block-sparse attention (§18.8.1): a CSR table lists, for each query block
    of ``block`` rows, the key blocks it attends to (row_ptr [nqb + 1],
    col_idx [nnz], strictly increasing within a row); key j is visible to
    query i iff j's block is listed for i's block (and, causal, j <= i).
    Unlisted blocks contribute nothing.  A row that sees no key gets O = 0 and
    LSE = -inf.  One table serves every batch entry and head.
  * paged, variable-length decode: a sequence's logical KV row r lives in the
    physical page block_table[b, r // page_size], at row r % page_size
    (PagedAttention's page table, §18.8.2 part 3 and §18.8.3); each sequence
    attends over its own first seqlens[b] rows, non-causally, which is the
    forward above applied to the gathered rows.

Large inputs are processed in blocks of whole query rows; every row's softmax
is still complete inside one block, so this is the plain definition, not a
tiling of it.
"""

import numpy as np

NEG_INF = -np.inf


def _f64(x):
    """Widen any array-like (numpy, or a torch tensor via numpy()) to float64."""
    if hasattr(x, "detach"):  # torch tensor: bf16 -> fp32 -> fp64 is exact
        import torch  # local import: the oracle itself does not need torch

        x = x.detach().to("cpu", torch.float32).numpy()
    return np.asarray(x, dtype=np.float64)


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, N, H, d]")
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv (grouped-query attention)")
    return B, Nq, Nk, Hq, Hkv, d


def causal_mask(rows, Nk):
    """Boolean matrix, True where key j is NOT visible to query row i (j > i).

    "第18章" §18.2.2: M_ij = -inf for j > i (top-left aligned; the causal
    configurations all have Nq == Nk).
    """
    rows = np.asarray(rows)
    return np.arange(Nk)[None, :] > rows[:, None]


def window_mask(rows, Nk, left, right):
    """Boolean matrix, True where key j is outside query row i's window
    [i - left, i + right] (a negative or None bound is unbounded)."""
    rows = np.asarray(rows)[:, None]
    j = np.arange(Nk)[None, :]
    out = np.zeros((rows.shape[0], Nk), dtype=bool)
    if left is not None and left >= 0:
        out |= j < rows - left
    if right is not None and right >= 0:
        out |= j > rows + right
    return out


def _scores(Qr, Kh, scale, rows, causal, window=None):
    S = scale * (Qr @ Kh.T)
    if causal:
        S = np.where(causal_mask(rows, Kh.shape[0]), NEG_INF, S)
    if window is not None:
        S = np.where(window_mask(rows, Kh.shape[0], *window), NEG_INF, S)
    return S


def _softmax_rows(S):
    """Safe softmax of each row (§18.4.2 'Safe Softmax'): max, exp, normalise."""
    m = S.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row sees no key (fully masked row)")
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    return E / l, m[:, 0], l[:, 0]


def attention_forward(q, k, v, scale, causal=False, row_block=2048, heads=None, rows=None, window=None):
    """Plain attention forward.  Returns (O [B,Nq,Hq,d], LSE [B,Hq,Nq]).

    ``window`` = (left, right) restricts query i to keys [i - left, i + right].

    ``heads`` (list of (b, h)) and ``rows`` (array of query rows) restrict which
    outputs are computed; entries not computed are NaN.  Restriction only skips
    rows: each computed row is the full definition.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    if (causal or window is not None) and Nq != Nk:
        raise ValueError("causal and windowed attention are defined here for Nq == Nk only")
    g = Hq // Hkv
    o = np.full((B, Nq, Hq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    all_rows = np.arange(Nq) if rows is None else np.asarray(rows)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]):
        kv = h // g
        Kh, Vh = k[b, :, kv, :], v[b, :, kv, :]
        for r0 in range(0, len(all_rows), row_block):
            rr = all_rows[r0:r0 + row_block]
            S = _scores(q[b, rr, h, :], Kh, scale, rr, causal, window)
            P, m, l = _softmax_rows(S)
            o[b, rr, h, :] = P @ Vh
            lse[b, h, rr] = m + np.log(l)
    return o, lse


def attention_backward(q, k, v, do, scale, causal=False, row_block=1024, heads=None, rows=None, window=None):
    """Plain attention backward with S and P materialised.

    Returns (dQ [B,Nq,Hq,d], dK [B,Nk,Hkv,d], dV [B,Nk,Hkv,d]).  With ``heads``
    given, only those query heads contribute (dQ of other heads is NaN and dK/dV
    hold only the listed heads' contributions).  With ``rows`` given, only those
    query rows are processed: dQ of other rows is NaN and dK/dV hold the sum of
    the listed rows' contributions (dK and dV are sums over query rows).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("dO must have the shape of O")
    if (causal or window is not None) and Nq != Nk:
        raise ValueError("causal and windowed attention are defined here for Nq == Nk only")
    g = Hq // Hkv
    dq = np.full(q.shape, np.nan)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]):
        kv = h // g
        Kh, Vh = k[b, :, kv, :], v[b, :, kv, :]
        all_rows = np.arange(Nq) if rows is None else np.asarray(rows)
        for r0 in range(0, len(all_rows), row_block):
            rr = all_rows[r0:r0 + row_block]
            Qr, dOr = q[b, rr, h, :], do[b, rr, h, :]
            S = _scores(Qr, Kh, scale, rr, causal, window)
            P, _, _ = _softmax_rows(S)
            dv[b, :, kv, :] += P.T @ dOr                 # dV = P^T dO
            dP = dOr @ Vh.T                              # dP = dO V^T
            D = np.sum(P * dP, axis=1, keepdims=True)    # D = rowsum(P o dP), full row
            dS = P * (dP - D)                            # softmax Jacobian
            dq[b, rr, h, :] = scale * (dS @ Kh)          # dQ = scale dS K
            dk[b, :, kv, :] += scale * (dS.T @ Qr)       # dK = scale dS^T Q
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, scale, causal, b, h, q_rows, k_rows, row_block=1024, window=None):
    """Backward of one query head (b, h), returning only sampled output rows.

    Returns (dQ[q_rows], dK_h[k_rows], dV_h[k_rows]) where dK_h/dV_h are the
    contributions of head h alone (sum them over a group for grouped heads).
    The full rows of S, P, dP and dS are formed exactly as in
    ``attention_backward``; only the rows kept at the end differ.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    kv = h // (Hq // Hkv)
    Kh, Vh = k[b, :, kv, :], v[b, :, kv, :]
    q_rows, k_rows = np.asarray(q_rows), np.asarray(k_rows)
    dq = np.zeros((len(q_rows), d))
    dk = np.zeros((len(k_rows), d))
    dv = np.zeros((len(k_rows), d))
    pos = {int(r): i for i, r in enumerate(q_rows)}
    for r0 in range(0, Nq, row_block):
        rr = np.arange(r0, min(Nq, r0 + row_block))
        Qr, dOr = q[b, rr, h, :], do[b, rr, h, :]
        S = _scores(Qr, Kh, scale, rr, causal, window)
        P, _, _ = _softmax_rows(S)
        dP = dOr @ Vh.T
        D = np.sum(P * dP, axis=1, keepdims=True)
        dS = P * (dP - D)
        dv += P[:, k_rows].T @ dOr
        dk += scale * (dS[:, k_rows].T @ Qr)
        for i, r in enumerate(rr):
            if int(r) in pos:
                dq[pos[int(r)]] = scale * (dS[i] @ Kh)
    return dq, dk, dv


def tiled_forward_head(Qh, Kh, Vh, scale, block_r, block_c, causal=False):
    """One head of the tiled forward with online softmax, in the pages' order.

    "第18章" §18.4.1 (outer loop over Q blocks of B_r rows, inner loop over K/V
    blocks of B_c rows, running state m, l, O) and §18.4.2 (online update:
    m_new = max(m, m~), l_new = e^{m-m_new} l + e^{m~-m_new} l~, and the output
    rescaled by the same factors; final O / l).  Block sizes may be anything;
    the result must equal the plain definition (the theorem of §18.4.2).
    Returns (O [Nq, d], LSE [Nq]).
    """
    Qh, Kh, Vh = _f64(Qh), _f64(Kh), _f64(Vh)
    Nq, d = Qh.shape
    Nk = Kh.shape[0]
    O = np.zeros((Nq, d))
    LSE = np.zeros(Nq)
    for i0 in range(0, Nq, block_r):
        rows = np.arange(i0, min(Nq, i0 + block_r))
        Qi = Qh[rows]
        m = np.full(len(rows), NEG_INF)
        l = np.zeros(len(rows))
        Oi = np.zeros((len(rows), d))
        for j0 in range(0, Nk, block_c):
            cols = np.arange(j0, min(Nk, j0 + block_c))
            Sij = scale * (Qi @ Kh[cols].T)
            if causal:
                Sij = np.where(cols[None, :] > rows[:, None], NEG_INF, Sij)
            m_tilde = Sij.max(axis=1)
            live = np.isfinite(m_tilde)        # rows with at least one visible key here
            safe_mt = np.where(live, m_tilde, 0.0)
            P_tilde = np.where(live[:, None], np.exp(Sij - safe_mt[:, None]), 0.0)
            l_tilde = P_tilde.sum(axis=1)
            m_new = np.maximum(m, m_tilde)
            a_old = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0)
            a_new = np.where(live, np.exp(m_tilde - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0)
            l = a_old * l + a_new * l_tilde
            Oi = a_old[:, None] * Oi + a_new[:, None] * (P_tilde @ Vh[cols])
            m = m_new
        O[rows] = Oi / l[:, None]
        LSE[rows] = m + np.log(l)
    return O, LSE


def tiled_forward_head_conditional(Qh, Kh, Vh, scale, block_r, block_c, threshold, causal=False):
    """One head of the tiled forward with conditional rescaling.

    "CMU 11-868 L21" notes on FA4: a variant of the online softmax that skips
    most rescalings.  Each row keeps a reference r in place of the running max;
    a new block's row max m~ replaces it only when m~ > r + threshold
    (``threshold`` in log2 units, i.e. r moves when a probability would exceed
    2^threshold).  Each block contributes P~ = exp(S - r_new) with
    r_new = m~ if it moved, else r; when r moves, l and O are rescaled by
    exp(r - r_new), as in the §18.4.2 update.  Final O / l and LSE = r + ln l.
    In exact arithmetic this is the plain definition for any threshold >= 0
    (the rescaling identity holds for any reference, not only the max).
    Returns (O [Nq, d], LSE [Nq], rescalings, p_max): rescalings counts the
    (row, block) steps after a row's first visible block in which r moved;
    p_max is the largest P~ entry seen (at most 2^threshold).
    """
    Qh, Kh, Vh = _f64(Qh), _f64(Kh), _f64(Vh)
    Nq, d = Qh.shape
    Nk = Kh.shape[0]
    tau = threshold * np.log(2.0)  # the scores are in natural-log units
    O = np.zeros((Nq, d))
    LSE = np.zeros(Nq)
    rescalings, p_max = 0, 0.0
    for i0 in range(0, Nq, block_r):
        rows = np.arange(i0, min(Nq, i0 + block_r))
        Qi = Qh[rows]
        r = np.full(len(rows), NEG_INF)
        l = np.zeros(len(rows))
        Oi = np.zeros((len(rows), d))
        for j0 in range(0, Nk, block_c):
            cols = np.arange(j0, min(Nk, j0 + block_c))
            Sij = scale * (Qi @ Kh[cols].T)
            if causal:
                Sij = np.where(cols[None, :] > rows[:, None], NEG_INF, Sij)
            m_tilde = Sij.max(axis=1)
            move = m_tilde > r + tau                     # -inf + tau stays -inf: a first visible block moves r
            rescalings += int(np.sum(move & np.isfinite(r)))
            r_new = np.where(move, m_tilde, r)
            seen = np.isfinite(r_new)
            base = np.where(seen, r_new, 0.0)
            alpha = np.where(np.isfinite(r), np.exp(r - base), 0.0)
            P_tilde = np.where(seen[:, None], np.exp(Sij - base[:, None]), 0.0)
            if P_tilde.size:
                p_max = max(p_max, float(P_tilde.max()))
            l = alpha * l + P_tilde.sum(axis=1)
            Oi = alpha[:, None] * Oi + P_tilde @ Vh[cols]
            r = r_new
        O[rows] = Oi / l[:, None]
        LSE[rows] = r + np.log(l)
    return O, LSE, rescalings, p_max


def two_block_output(Qh, K1, V1, K2, V2, scale):
    """Two-block rescaling of lecture slide 12, with exp taken without a max.

    l1 = rowsum(exp(S1)), O1 = exp(S1) V1 / l1; l2 = l1 + rowsum(exp(S2));
    O2 = (l1 / l2) O1 + exp(S2) V2 / l2.  Only for small scores (no max shift).
    """
    Qh, K1, V1, K2, V2 = map(_f64, (Qh, K1, V1, K2, V2))
    A1 = np.exp(scale * (Qh @ K1.T))
    A2 = np.exp(scale * (Qh @ K2.T))
    l1 = A1.sum(axis=1, keepdims=True)
    O1 = (A1 @ V1) / l1
    l2 = l1 + A2.sum(axis=1, keepdims=True)
    return (l1 / l2) * O1 + (A2 @ V2) / l2


def decode_partials(q, k, v, scale, splits, heads=None):
    """FlashDecoding step 2 ("第18章" §18.8.2): per KV split, local statistics.

    ``splits`` is a list of (start, end) key ranges.  Returns (m, l, O_t) with
    shapes [B, Hq, Nq, T], [B, Hq, Nq, T] and [B, Hq, Nq, T, d], where O_t is the
    unnormalised local output sum_j e^{s_j - m_t} v_j.  An empty split has
    m = -inf, l = 0, O_t = 0.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    T = len(splits)
    m = np.full((B, Hq, Nq, T), NEG_INF)
    l = np.zeros((B, Hq, Nq, T))
    Ot = np.zeros((B, Hq, Nq, T, d))
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]):
        kv = h // g
        for t, (s0, s1) in enumerate(splits):
            if s1 <= s0:
                continue
            s = scale * (q[b, :, h, :] @ k[b, s0:s1, kv, :].T)   # [Nq, keys]
            mt = s.max(axis=1)
            e = np.exp(s - mt[:, None])
            m[b, h, :, t] = mt
            l[b, h, :, t] = e.sum(axis=1)
            Ot[b, h, :, t, :] = e @ v[b, s0:s1, kv, :]
    return m, l, Ot


def decode_combine(m, l, Ot):
    """FlashDecoding step 3: O = sum_t O_t e^{m_t - m} / sum_t l_t e^{m_t - m}.

    Returns (O [B, Hq, Nq, d], LSE [B, Hq, Nq]) with LSE = m + ln sum_t l_t e^{m_t-m}.
    """
    mg = m.max(axis=-1)
    w = np.where(np.isfinite(m), np.exp(m - mg[..., None]), 0.0)
    den = np.sum(l * w, axis=-1)
    O = np.sum(Ot * w[..., None], axis=-2) / den[..., None]
    return O, mg + np.log(den)


def _seq_bounds(cu):
    cu = np.asarray(cu, dtype=np.int64)
    if cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    return cu


def attention_varlen_forward(q, k, v, cu_q, cu_k, scale, causal=False):
    """Packed variable-length forward: each sequence is plain attention over its own
    rows.  q [total_q, Hq, d], k/v [total_k, Hkv, d]; returns (O [total_q, Hq, d],
    LSE [Hq, total_q]).  Causal needs equal query and key lengths per sequence."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _seq_bounds(cu_q), _seq_bounds(cu_k)
    O = np.zeros(q.shape)
    LSE = np.zeros((q.shape[1], q.shape[0]))
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        if k1 == k0:
            raise ValueError("a sequence with queries but no keys has no attention")
        Ob, Lb = attention_forward(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale, causal)
        O[q0:q1], LSE[:, q0:q1] = Ob[0], Lb[0]
    return O, LSE


def attention_varlen_backward(q, k, v, do, cu_q, cu_k, scale, causal=False):
    """Gradients (dQ, dK, dV) of the packed forward, sequence by sequence; keys of a
    sequence with no queries get zero gradients."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cq, ck = _seq_bounds(cu_q), _seq_bounds(cu_k)
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        g = attention_backward(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], do[None, q0:q1], scale, causal)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


def block_mask_from_csr(row_ptr, col_idx, n_qblocks, n_kblocks):
    """Dense boolean [n_qblocks, n_kblocks] of the listed blocks; raises on a table
    that is not strictly increasing within rows or lists a block out of range."""
    row_ptr, col_idx = np.asarray(row_ptr, dtype=np.int64), np.asarray(col_idx, dtype=np.int64)
    if len(row_ptr) != n_qblocks + 1 or row_ptr[0] != 0 or np.any(np.diff(row_ptr) < 0):
        raise ValueError("row_ptr must have one entry per query block plus one, from 0, non-decreasing")
    M = np.zeros((n_qblocks, n_kblocks), dtype=bool)
    for i in range(n_qblocks):
        cols = col_idx[row_ptr[i]:row_ptr[i + 1]]
        if np.any(np.diff(cols) <= 0) or np.any(cols < 0) or np.any(cols >= n_kblocks):
            raise ValueError("column indices must be strictly increasing and within range")
        M[i, cols] = True
    return M


def attention_blocksparse_forward(q, k, v, row_ptr, col_idx, scale, causal=False, block=128):
    """Block-sparse forward: O [B, Nq, Hq, d], LSE [B, Hq, Nq].  Plain definition with
    the element mask taken from the listed blocks; rows that see no key get O = 0,
    LSE = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    if causal and Nq != Nk:
        raise ValueError("causal attention is defined here for Nq == Nk only")
    M = block_mask_from_csr(row_ptr, col_idx, -(-Nq // block), -(-Nk // block))
    visible = np.repeat(np.repeat(M, block, axis=0), block, axis=1)[:Nq, :Nk]
    if causal:
        visible &= ~causal_mask(np.arange(Nq), Nk)
    g = Hq // Hkv
    O = np.zeros((B, Nq, Hq, d))
    LSE = np.full((B, Hq, Nq), NEG_INF)
    seen = visible.any(axis=1)
    for b in range(B):
        for h in range(Hq):
            S = np.where(visible, scale * (q[b, :, h, :] @ k[b, :, h // g, :].T), NEG_INF)
            m = np.where(seen, S.max(axis=1), 0.0)
            E = np.where(visible, np.exp(S - m[:, None]), 0.0)
            l = E.sum(axis=1)
            O[b, seen, h, :] = (E[seen] @ v[b, :, h // g, :]) / l[seen, None]
            LSE[b, h, seen] = m[seen] + np.log(l[seen])
    return O, LSE


def attention_blocksparse_backward(q, k, v, do, row_ptr, col_idx, scale, causal=False, block=128):
    """Gradients (dQ, dK, dV) of the block-sparse forward: the plain backward with
    S = -inf outside the visible pairs (P = 0 there); rows that see no key
    contribute nothing."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    if causal and Nq != Nk:
        raise ValueError("causal attention is defined here for Nq == Nk only")
    M = block_mask_from_csr(row_ptr, col_idx, -(-Nq // block), -(-Nk // block))
    visible = np.repeat(np.repeat(M, block, axis=0), block, axis=1)[:Nq, :Nk]
    if causal:
        visible &= ~causal_mask(np.arange(Nq), Nk)
    seen = visible.any(axis=1)
    g = Hq // Hkv
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            S = np.where(visible, scale * (q[b, :, h, :] @ k[b, :, kv, :].T), NEG_INF)
            m = np.where(seen, S.max(axis=1), 0.0)
            E = np.where(visible, np.exp(S - m[:, None]), 0.0)
            P = E / np.where(seen, E.sum(axis=1), 1.0)[:, None]
            dO = do[b, :, h, :]
            dv[b, :, kv, :] += P.T @ dO
            dP = dO @ v[b, :, kv, :].T
            D = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dq[b, :, h, :] = scale * dS @ k[b, :, kv, :]
            dk[b, :, kv, :] += scale * dS.T @ q[b, :, h, :]
    return dq, dk, dv


def attention_blocksparse_backward_sampled(q, k, v, do, row_ptr, col_idx, scale, causal, b, h, q_rows, k_rows,
                                           block=128):
    """Sampled rows of the block-sparse backward of one query head (b, h).

    Returns (dQ[q_rows], dK_h[k_rows], dV_h[k_rows]), dK_h/dV_h being head h's
    contributions.  The definition of ``attention_blocksparse_backward`` taken
    one query block at a time over the key blocks it lists (P is 0 elsewhere,
    so the other key blocks add nothing): with K_L, V_L the listed keys,
        P = softmax(scale Q_i K_L^T) (causal: keys after the row masked),
        dP = dO_i V_L^T, D = rowsum(P o dP), dS = P o (dP - D),
        dQ_i = scale dS K_L, dK_L += scale dS^T Q_i, dV_L += P^T dO_i.
    Query blocks that hold no sampled row and list no block of a sampled key
    row are skipped."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Nq, Nk, Hq, Hkv, d = _check_shapes(q, k, v)
    if causal and Nq != Nk:
        raise ValueError("causal attention is defined here for Nq == Nk only")
    nqb, nkb = -(-Nq // block), -(-Nk // block)
    M = block_mask_from_csr(row_ptr, col_idx, nqb, nkb)
    kv = h // (Hq // Hkv)
    q_rows, k_rows = np.asarray(q_rows), np.asarray(k_rows)
    dq = np.zeros((len(q_rows), d))
    dk = np.zeros((len(k_rows), d))
    dv = np.zeros((len(k_rows), d))
    k_blocks = set((k_rows // block).tolist())
    q_blocks = set((q_rows // block).tolist())
    for i in range(nqb):
        listed = np.flatnonzero(M[i])
        if len(listed) == 0 or not (i in q_blocks or k_blocks & set(listed.tolist())):
            continue
        rows = np.arange(i * block, min(Nq, (i + 1) * block))
        keys = np.concatenate([np.arange(j * block, min(Nk, (j + 1) * block)) for j in listed])
        vis = np.ones((len(rows), len(keys)), dtype=bool)
        if causal:
            vis &= keys[None, :] <= rows[:, None]
        seen = vis.any(axis=1)
        S = np.where(vis, scale * (q[b, rows, h, :] @ k[b, keys, kv, :].T), NEG_INF)
        m = np.where(seen, S.max(axis=1), 0.0)
        E = np.where(vis, np.exp(S - m[:, None]), 0.0)
        P = E / np.where(seen, E.sum(axis=1), 1.0)[:, None]
        dO = do[b, rows, h, :]
        dP = dO @ v[b, keys, kv, :].T
        D = (P * dP).sum(axis=1, keepdims=True)
        dS = P * (dP - D)
        for t, r in enumerate(q_rows):
            if r // block == i:
                dq[t] = scale * (dS[r - i * block] @ k[b, keys, kv, :])
        pos = {int(key): c for c, key in enumerate(keys)}
        for t, key in enumerate(k_rows):
            c = pos.get(int(key))
            if c is not None:
                dk[t] += scale * (dS[:, c] @ q[b, rows, h, :])
                dv[t] += P[:, c] @ dO
    return dq, dk, dv


def gather_paged(cache, block_table, b, length):
    """Logical rows [0, length) of sequence b from a paged cache [pages, page_size, H, d]:
    row r is at page block_table[b, r // page_size], row r % page_size."""
    cache = np.asarray(cache)
    page_size = cache.shape[1]
    r = np.arange(length)
    return cache[np.asarray(block_table)[b, r // page_size], r % page_size]


def attention_decode_paged(q, k_cache, v_cache, block_table, seqlens, scale):
    """Decode over a paged, variable-length KV cache.

    q [B, Nq, Hq, d]; k_cache, v_cache [pages, page_size, Hkv, d]; block_table
    [B, max_pages] int; seqlens [B] int >= 1.  Sequence b attends, non-causally,
    over its own first seqlens[b] logical KV rows.  Returns (O [B, Nq, Hq, d],
    LSE [B, Hq, Nq]).
    """
    q = _f64(q)
    kc, vc = _f64(k_cache), _f64(v_cache)
    B, Nq, Hq, d = q.shape
    O = np.zeros((B, Nq, Hq, d))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        L = int(seqlens[b])
        kb = gather_paged(kc, block_table, b, L)[None]
        vb = gather_paged(vc, block_table, b, L)[None]
        Ob, LSEb = attention_forward(q[b:b + 1], kb, vb, scale, causal=False)
        O[b], LSE[b] = Ob[0], LSEb[0]
    return O, LSE


def flops_forward(B, Hq, Nq, Nk, d, causal):
    """Counted forward FLOPs: two matmuls of 2*Nq*Nk*d each per head, halved for causal.

    "第18章" §18.2.3 (about 4N^2 d for the two products) and §18.5.2 (causal
    roughly halves it).  Softmax FLOPs are not counted.
    """
    f = 4.0 * B * Hq * Nq * Nk * d
    return f / 2 if causal else f


def flops_backward(B, Hq, Nq, Nk, d, causal):
    """Counted backward FLOPs: 2.5x the forward (five matmuls instead of two)."""
    return 2.5 * flops_forward(B, Hq, Nq, Nk, d, causal)
