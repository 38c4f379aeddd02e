// Integer plans shared by the host API and the kernels: causal tile classes,
// visited tile ranges, the longest-first work-unit orders and the decode
// splits.  One definition serves both sides, so what the host reports is what
// the kernels do.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int TILE = 128;  // query-tile rows and key-tile rows

FA_HD int cdiv(int a, int b) { return (a + b - 1) / b; }
FA_HD int imin(int a, int b) { return a < b ? a : b; }
FA_HD int imax(int a, int b) { return a > b ? a : b; }

// Keys visible to query row i: i - wl <= j <= i + wr.  Causal attention is the
// band with wr = 0 (and wl unbounded); a sliding window sets both; UNBOUNDED
// (larger than any sequence) leaves a side open.
constexpr int UNBOUNDED = 1 << 29;

struct Dims {
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int wl, wr;  // band of visible keys around each row (causal folded into wr)
  // Packed variable-length sequences (cu_q == nullptr: dense [B, N, H, d]).
  // Sequence b is rows cu_q[b] .. cu_q[b+1]-1 of Q (cu_k likewise of K, V),
  // tensors [total, H, d]; Nq and Nk then hold the longest lengths, which size
  // the work-unit grid, and every unit works on its own sequence's lengths.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
};

#ifdef __CUDACC__
// The rows a work unit of batch entry b sees: its own lengths (in `s`) and
// where they start in the tensors.  Dense: b's rows from 0, TMA batch
// coordinate b.  Packed: rows cu[b].., batch coordinate 0.  `ok` is false for
// lengths the cu arrays cannot hold (not within [0, total], decreasing, longer
// than the grid's Nq / Nk, queries without keys, or unequal lengths under a
// causal mask); such a sequence is given no rows.
struct SeqRows {
  Dims s;
  int qoff, koff, tb;
  bool ok;
};

template <bool VL>  // VL: packed sequences (else the dense view, at no cost)
__device__ __forceinline__ SeqRows seq_rows(const Dims& d, int b) {
  SeqRows r{d, 0, 0, b, true};
  if (!VL) return r;
  const int q0 = __ldg(d.cu_q + b), q1 = __ldg(d.cu_q + b + 1);
  const int k0 = __ldg(d.cu_k + b), k1 = __ldg(d.cu_k + b + 1);
  r.ok = 0 <= q0 && q0 <= q1 && q1 <= d.total_q && 0 <= k0 && k0 <= k1 && k1 <= d.total_k &&
         q1 - q0 <= d.Nq && k1 - k0 <= d.Nk && (q1 == q0 || k1 > k0) && (!d.causal || q1 - q0 == k1 - k0);
  r.s.Nq = r.ok ? q1 - q0 : 0;
  r.s.Nk = r.ok ? k1 - k0 : 0;
  r.qoff = r.ok ? q0 : 0;
  r.koff = r.ok ? k0 : 0;
  r.tb = 0;
  return r;
}

// Work plan of packed sequences, built on the device for each call (see
// launch_varlen_plan): units with work only, longest first.  A unit has a
// level (forward: the query-tile pair; dQ: the query tile; dK/dV: the key tile
// counted from the sequence's end) and levels are handed out from the highest
// down; within a level come the sequences long enough to have it, in
// descending order of their level count, each with all its heads (adjacent,
// so heads sharing a K/V head stay together).  Layout (ints): [0] units,
// [1] levels n, [4 .. 4+n] first unit of each level, highest level first
// (the last entry = units), then [B] the sequences in order.
__device__ __forceinline__ void plan_unit(const int* plan, int heads, int u, int& b, int& h, int& level) {
  const int nlev = __ldg(plan + 1);
  const int* ls = plan + 4;
  int lo = 0, hi = nlev;  // ls[lo] <= u < ls[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ls + mid) <= u)
      lo = mid;
    else
      hi = mid;
  }
  const int r = u - __ldg(ls + lo);
  b = __ldg(ls + nlev + 1 + r / heads);
  h = r % heads;
  level = nlev - 1 - lo;
}
#endif

// ints a varlen plan with `levels` levels over B sequences takes
FA_HD int varlen_plan_ints(int levels, int B) { return 4 + levels + 1 + B; }

FA_HD bool banded(const Dims& s) { return s.wl < UNBOUNDED || s.wr < UNBOUNDED; }

// Which masking a kernel instantiation handles: none, causal (j <= i only; the
// last visited tile is the only partial one), or a general band.
constexpr int MASK_NONE = 0, MASK_CAUSAL = 1, MASK_BAND = 2;
FA_HD int mask_kind(const Dims& s) {
  if (s.wl < UNBOUNDED || (!s.causal && s.wr < UNBOUNDED)) return MASK_BAND;
  return s.causal ? MASK_CAUSAL : MASK_NONE;
}

// "第18章 FlashAttention" §18.5.2: a block of rows [qs, qe) and keys [ks, ke)
// is fully masked, fully visible or partial; under j <= i the first happens
// when ks > qe-1 and the second when ke-1 <= qs.  The same test for the band
// i - wl <= j <= i + wr: no key of the block is visible to any row when the
// block lies right of the last row's reach (ks > qe-1 + wr) or left of the first
// row's (ke-1 < qs - wl); every key is visible to every row when the block's
// corners are (ke-1 <= qs + wr and ks >= qe-1 - wl).  0 = skip, 1 = full,
// 2 = partial.  (64-bit: wl and wr may be UNBOUNDED.)
FA_HD int band_class(int qs, int qe, int ks, int ke, int wl, int wr) {
  const long long qs_ = qs, qe_ = qe, ks_ = ks, ke_ = ke;
  if (ks_ > qe_ - 1 + wr || ke_ - 1 < qs_ - wl) return 0;
  if (ke_ - 1 <= qs_ + wr && ks_ >= qe_ - 1 - wl) return 1;
  return 2;
}

FA_HD int tile_class(const Dims& s, int qt, int kt) {
  if (!banded(s)) return 1;
  return band_class(qt * TILE, imin(s.Nq, (qt + 1) * TILE), kt * TILE, imin(s.Nk, (kt + 1) * TILE), s.wl, s.wr);
}

FA_HD int q_tiles(const Dims& s) { return cdiv(s.Nq, TILE); }
FA_HD int k_tiles(const Dims& s) { return cdiv(s.Nk, TILE); }

// Key tiles visited by query tile qt: the range [lo, hi) of tiles holding a key
// some row of the tile can see.  Under j <= i that is a prefix ending at the
// tile of the last row (§18.5.2's bound ceil((q_start + B_r) / B_c), clipped to
// the sequence); under a band it also starts at the first row's reach.
FA_HD void kv_range(const Dims& s, int qt, int& lo, int& hi) {
  const int nk = k_tiles(s);
  const long long first = static_cast<long long>(qt) * TILE - s.wl;
  const long long last = static_cast<long long>(imin(s.Nq, (qt + 1) * TILE)) - 1 + s.wr;
  lo = first <= 0 ? 0 : static_cast<int>(first / TILE);
  hi = last >= static_cast<long long>(nk) * TILE ? nk : static_cast<int>(last / TILE) + 1;
}

FA_HD int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Key tiles that query tile qt sees in full are [lo, hi] (a superset of its
// visited range may result; callers intersect): every row of [qs, qe) must
// reach the tile's first key (kt*TILE >= qe-1 - wl) and its last key
// (kt*TILE + TILE-1 <= qs + wr).  Ragged sequence ends are not counted here.
FA_HD void kv_full_range(const Dims& s, int qt, int& lo, int& hi) {
  const int qs = qt * TILE, qe = imin(s.Nq, qs + TILE);
  lo = imax(0, floor_div(qe - 1 - s.wl + TILE - 1, TILE));
  hi = floor_div(qs + s.wr - (TILE - 1), TILE);
}

// Query tiles whose rows all see every key of key tile kt are [lo, hi]: rows
// j - wr .. j + wl see key j, so a query tile is full for keys [ks, ke) when
// its first row reaches ke-1 - wr and its last row at most ks + wl.
FA_HD void q_full_range(const Dims& s, int kt, int& lo, int& hi) {
  const int ks = kt * TILE, ke = imin(s.Nk, ks + TILE);
  lo = imax(0, floor_div(ke - 1 - s.wr + TILE - 1, TILE));
  hi = floor_div(ks + s.wl - (TILE - 1), TILE);
}

// Query tiles visiting key tile kt: the range [lo, hi) of tiles holding a row
// that sees some key of the tile (rows j - wr .. j + wl see key j).
FA_HD void q_range(const Dims& s, int kt, int& lo, int& hi) {
  const int nq = q_tiles(s);
  const long long first = static_cast<long long>(kt) * TILE - s.wr;
  const long long last = static_cast<long long>(imin(s.Nk, (kt + 1) * TILE)) - 1 + s.wl;
  lo = first <= 0 ? 0 : static_cast<int>(first / TILE);
  hi = last >= static_cast<long long>(nq) * TILE ? nq : static_cast<int>(last / TILE) + 1;
}

// ---- forward units: (b, h, p) = query tiles 2p and 2p+1 of head h ------------
// Longest first ("CMU 11-868 L21" notes, slides 27-46): causal units cost
// more as p grows, so they are handed out with p descending; equal costs keep
// (b, h) order, which also keeps the heads sharing a K/V head adjacent.
FA_HD int fwd_pairs(const Dims& s) { return cdiv(q_tiles(s), 2); }
FA_HD int fwd_units(const Dims& s) { return s.B * s.Hq * fwd_pairs(s); }

FA_HD void fwd_unit(const Dims& s, int u, int& b, int& h, int& p) {
  const int P = fwd_pairs(s), BH = s.B * s.Hq;
  int bh;
  if (s.causal) {
    bh = u % BH;
    p = P - 1 - u / BH;
  } else {
    bh = u / P;
    p = u % P;
  }
  b = bh / s.Hq;
  h = bh % s.Hq;
}

// The unit index of (b, h, p): the inverse of fwd_unit.
FA_HD int fwd_unit_index(const Dims& s, int b, int h, int p) {
  const int P = fwd_pairs(s), BH = s.B * s.Hq, bh = b * s.Hq + h;
  return s.causal ? (P - 1 - p) * BH + bh : bh * P + p;
}

// ---- dK/dV units: (b, kvh, kt) -------------------------------------------------
FA_HD int dkdv_units(const Dims& s) { return s.B * s.Hkv * k_tiles(s); }

FA_HD void dkdv_unit(const Dims& s, int u, int& b, int& kvh, int& kt) {
  const int nk = k_tiles(s), BK = s.B * s.Hkv;
  int bk;
  if (s.causal) {  // early key tiles see the most query tiles
    bk = u % BK;
    kt = u / BK;
  } else {
    bk = u / nk;
    kt = u % nk;
  }
  b = bk / s.Hkv;
  kvh = bk % s.Hkv;
}

// ---- dQ units: (b, h, qt) --------------------------------------------------------
FA_HD int dq_units(const Dims& s) { return s.B * s.Hq * q_tiles(s); }

FA_HD void dq_unit(const Dims& s, int u, int& b, int& h, int& qt) {
  const int nq = q_tiles(s), BH = s.B * s.Hq;
  int bh;
  if (s.causal) {
    bh = u % BH;
    qt = nq - 1 - u / BH;
  } else {
    bh = u / nq;
    qt = u % nq;
  }
  b = bh / s.Hq;
  h = bh % s.Hq;
}

// ---- decode splits ("第18章" §18.8.2): whole tiles, none empty -------------------
FA_HD int decode_chunk(int Nk, int S) { return cdiv(cdiv(Nk, TILE), S) * TILE; }
FA_HD int decode_nsplits(int Nk, int S) { return cdiv(Nk, decode_chunk(Nk, S)); }

}  // namespace fa
