"""Integer plans of the attention hot path, written out plainly (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Pure Python integers.

  * causal tile classes -- "第18章 FlashAttention" §18.5.2: a (Q block, K block)
    pair is fully visible, fully masked (skipped) or partial (masked element by
    element).  Fig. 18-20 shows the 3x3 case.
  * sliding-window tile classes -- the same three classes under the predicate
    i - left <= j <= i + right (§18.8.1's block-sparse loop skips the blocks no
    row of the query block can see; a sliding window is its banded case).
  * longest-first order and greedy list scheduling -- "CMU 11-868 L21
    FlashAttention" notes, slides 27-46 (LPT: schedule the longest work first;
    worked example with 2 batches on 3 SMs: in-order loads [9, 5, 6], longest
    first [7, 7, 6]).
  * decode split boundaries -- "第18章" §18.8.2: the KV cache is cut along its
    length into chunks, one per thread block; chunks are whole 128-key tiles.
"""

SKIP, FULL, PARTIAL = 0, 1, 2


def cdiv(a, b):
    return -(-a // b)


def causal_tile_class(q_start, q_end, k_start, k_end):
    """Class of the block rows [q_start, q_end) x keys [k_start, k_end) under j <= i.

    Fully masked when every key index exceeds every row index (k_start > q_end-1);
    fully visible when every key index is at most every row index
    (k_end-1 <= q_start); otherwise partial.
    """
    if k_start > q_end - 1:
        return SKIP
    if k_end - 1 <= q_start:
        return FULL
    return PARTIAL


def window_tile_class(q_start, q_end, k_start, k_end, left, right, causal):
    """Class of rows [q_start, q_end) x keys [k_start, k_end) under i - left <= j <= i + right
    (and j <= i when causal); a negative bound is unbounded.

    Skipped when no (row, key) pair is visible; full when every pair is; else partial.
    """
    if causal:
        right = 0 if right < 0 else min(right, 0)
    lo_ok = lambda i, j: left < 0 or j >= i - left       # noqa: E731
    hi_ok = lambda i, j: right < 0 or j <= i + right     # noqa: E731
    # visible pairs exist iff the band meets the rectangle: the smallest key any row can
    # see is q_start - left, the largest q_end - 1 + right
    if (right >= 0 and k_start > q_end - 1 + right) or (left >= 0 and k_end - 1 < q_start - left):
        return SKIP
    if lo_ok(q_end - 1, k_start) and hi_ok(q_start, k_end - 1):
        return FULL
    return PARTIAL


def tile_ranges(Nq, Nk, block, left, right, causal):
    """For each query tile, the half-open range of key tiles that are not skipped."""
    out = []
    for i in range(cdiv(Nq, block)):
        qs, qe = i * block, min(Nq, (i + 1) * block)
        vis = [j for j in range(cdiv(Nk, block))
               if window_tile_class(qs, qe, j * block, min(Nk, (j + 1) * block), left, right, causal) != SKIP]
        out.append((min(vis), max(vis) + 1) if vis else (0, 0))
    return out


def tile_classes(Nq, Nk, block_m, block_n, causal):
    """Matrix [ceil(Nq/bm)][ceil(Nk/bn)] of tile classes (all FULL if not causal)."""
    out = []
    for i in range(cdiv(Nq, block_m)):
        row = []
        for j in range(cdiv(Nk, block_n)):
            if not causal:
                row.append(FULL)
            else:
                row.append(causal_tile_class(i * block_m, min(Nq, (i + 1) * block_m),
                                             j * block_n, min(Nk, (j + 1) * block_n)))
        out.append(row)
    return out


def greedy_loads(costs, n_workers, longest_first):
    """Greedy list scheduling: each job, in turn, goes to the least-loaded worker.

    Ties go to the lowest worker index.  With ``longest_first`` the jobs are
    first sorted by cost, largest first (a stable sort), which is LPT.
    Returns the final load of each worker.
    """
    jobs = list(costs)
    if longest_first:
        jobs = sorted(jobs, key=lambda c: -c)
    loads = [0] * n_workers
    for c in jobs:
        w = min(range(n_workers), key=lambda i: (loads[i], i))
        loads[w] += c
    return loads


# -- work units and their longest-first order -------------------------------------
# A forward unit is (b, h, p): query tiles 2p and 2p+1 (128 rows each) of head h.
# Its cost is the number of 128-key tiles its loop visits.  Units are listed by
# cost, largest first; equal costs keep (b, h, p) order.

TILE = 128


def fwd_unit_cost(Nq, Nk, causal, p):
    """Key tiles visited by unit p: those not skipped for either of its query tiles."""
    nq_t, nk_t = cdiv(Nq, TILE), cdiv(Nk, TILE)
    tiles = [t for t in (2 * p, 2 * p + 1) if t < nq_t]
    return sum(1 for j in range(nk_t) if any(
        not causal or causal_tile_class(t * TILE, min(Nq, (t + 1) * TILE),
                                        j * TILE, min(Nk, (j + 1) * TILE)) != SKIP
        for t in tiles))


def fwd_unit_order(B, Hq, Nq, Nk, causal):
    pairs = cdiv(cdiv(Nq, TILE), 2)
    units = [(b, h, p) for b in range(B) for h in range(Hq) for p in range(pairs)]
    return sorted(units, key=lambda u: (-fwd_unit_cost(Nq, Nk, causal, u[2]), u))


def dkdv_unit_order(B, Hkv, Nq, Nk, causal):
    """dK/dV units (b, kvh, j): key tile j of KV head kvh; cost = query tiles visited."""
    nq_t, nk_t = cdiv(Nq, TILE), cdiv(Nk, TILE)

    def cost(j):
        if not causal:
            return nq_t
        return sum(1 for i in range(nq_t) if causal_tile_class(
            i * TILE, min(Nq, (i + 1) * TILE), j * TILE, min(Nk, (j + 1) * TILE)) != SKIP)

    units = [(b, kh, j) for b in range(B) for kh in range(Hkv) for j in range(nk_t)]
    return sorted(units, key=lambda u: (-cost(u[2]), u))


def dq_unit_order(B, Hq, Nq, Nk, causal):
    """dQ units (b, h, i): query tile i of head h; cost = key tiles visited."""
    nq_t, nk_t = cdiv(Nq, TILE), cdiv(Nk, TILE)

    def cost(i):
        if not causal:
            return nk_t
        return sum(1 for j in range(nk_t) if causal_tile_class(
            i * TILE, min(Nq, (i + 1) * TILE), j * TILE, min(Nk, (j + 1) * TILE)) != SKIP)

    units = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(nq_t)]
    return sorted(units, key=lambda u: (-cost(u[2]), u))


def decode_splits(Nk, num_splits):
    """Key ranges of the decode splits: whole 128-key tiles, none empty.

    chunk = ceil(ceil(Nk/128) / S) * 128 keys; split s covers
    [s*chunk, min((s+1)*chunk, Nk)); the number of splits is ceil(Nk / chunk),
    which can be below the requested S when Nk is short.
    """
    if Nk <= 0 or num_splits <= 0:
        raise ValueError("Nk and num_splits must be positive")
    chunk = cdiv(cdiv(Nk, TILE), num_splits) * TILE
    n = cdiv(Nk, chunk)
    return [(s * chunk, min((s + 1) * chunk, Nk)) for s in range(n)]
