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

struct Dims {
  int B, Hq, Hkv, Nq, Nk;
  int causal;
};

// "第18章 FlashAttention" §18.5.2: with rows [qs, qe) and keys [ks, ke) under
// the rule j <= i, the block is fully masked when ks > qe-1, fully visible
// when ke-1 <= qs, and partial otherwise.  0 = skip, 1 = full, 2 = partial.
FA_HD int causal_class(int qs, int qe, int ks, int ke) {
  if (ks > qe - 1) return 0;
  if (ke - 1 <= qs) return 1;
  return 2;
}

FA_HD int tile_class(const Dims& s, int qt, int kt) {
  if (!s.causal) return 1;
  return causal_class(qt * TILE, imin(s.Nq, (qt + 1) * TILE), kt * TILE, imin(s.Nk, (kt + 1) * TILE));
}

FA_HD int q_tiles(const Dims& s) { return cdiv(s.Nq, TILE); }
FA_HD int k_tiles(const Dims& s) { return cdiv(s.Nk, TILE); }

// Key tiles visited by query tile qt: a prefix [0, n).  Under j <= i key tile
// kt is visited iff its first key is at most the tile's last row (§18.5.2's
// bound ceil((q_start + B_r) / B_c), clipped to the sequence).
FA_HD int kv_tiles_for_q(const Dims& s, int qt) {
  const int nk = k_tiles(s);
  if (!s.causal) return nk;
  const int last_row = imin(s.Nq, (qt + 1) * TILE) - 1;
  return imin(nk, last_row / TILE + 1);
}

// Query tiles visited by key tile kt: a suffix [first, nq).
FA_HD int q_tile_begin(const Dims& s, int kt) {
  if (!s.causal) return 0;
  return (kt * TILE) / TILE;  // first query tile whose last row reaches key kt*TILE
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
