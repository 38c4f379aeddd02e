// Forward kernel: exact attention, tile by tile with an online softmax.
//
// Method ("第18章 FlashAttention" §18.4.1-§18.4.3; "CMU 11-868 L21" notes,
// slides 9-12 and the Algorithm-1 remark): each query tile keeps a running row
// max m and row sum l; every key tile's scores S = Q K^T are exponentiated
// against the running max, the partial output is rescaled when the max moves,
// and at the end O / l and LSE = m + ln l are written.  S and P never leave the
// chip.  Causal work skips key tiles above the diagonal and masks the diagonal
// tile element by element (§18.5.2).
//
// GB300 design (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer: claims work units (an atomic counter, longest
//               first), loads the two Q tiles of the unit and streams K_j, V_j
//               through a ring of shared-memory stages.
//   warp 1      MMA issuer (one thread) and TMEM owner: S_t = Q_t K_j^T and
//               O_t += P_t V_j with tcgen05.mma, accumulators in TMEM.
//   warps 4-7   softmax for query tile 0 of the unit (thread = row = TMEM lane)
//   warps 8-11  softmax for query tile 1
// Each softmax warp also writes its rows' output: O / l in 32-column boxes staged
// in shared memory and stored by the copy engine (TMA), so the warp only fills a
// 2 KB buffer per box and can start the next unit while the stores drain.
// The two query tiles share every K/V stage and ping-pong on the tensor core:
// while one warpgroup exponentiates S_0, the tensor core computes S_1 or P_0 V.
// TMEM (512 columns): S_0 [0,128) S_1 [128,256) O_0 [256,256+d) O_1 [256+d,256+2d);
// P_t is written as bf16 over the first 64 columns of S_t and read from TMEM by
// the P V product.
// FP8 instantiation ("第18章" §18.6.2): Q, K, V arrive as E4M3 codes with
// per-block scales for Q and K and one scale per head for V; S = Q K^T and O +=
// P V run as kind::f8f6f4 products (K = 32 per instruction), S is scaled by
// the product of the two block scales, the softmax stays in fp32, and P goes
// to TMEM as E4M3 on the scale its bound fixes (448 P, four codes per column);
// the epilogue applies V's scale with 1 / l.
// Block-sparse instantiation (§18.8.1): a CSR table lists the key tiles of each
// query tile.  Warp 2 turns a unit's two rows of the table into one list in
// shared memory (the union in key order, with a bit per query tile) and the
// other roles walk it: K/V of listed tiles only, S and P V of a query tile only
// at its own tiles.  Consumers release a unit's slot when the unit is done
// (the list lives there until then).
// The reference of the exponent is the running max.  By default (tau = 0) it
// is the exact row max so far: the dominant P of a nearly one-hot row is then
// exactly 1.0 in bf16, so O's error scales with the rest of the row, which keeps
// D = dO . O consistent in the backward.  The rescale of O is skipped for a warp
// whose 32 rows kept their reference.  Conditional rescaling (lecture notes,
// FA4: most rescalings skipped) is the opt-in tau > 0: the reference moves
// only when a tile's max exceeds it by more than tau (log2 units), so P may
// reach 2^tau and most tiles keep alpha = 1; O / l is still exact, but the
// dominant P is rounded (to bf16, or as E4M3 with P's scale 2^tau / 448).
#include <math.h>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float LN2 = 0.69314718055994530942f;
constexpr float LOG2_448 = 8.8073549220576041f;  // P is quantised as 448 P = 2^(x - m + log2 448)

template <int D, bool F8 = false, bool SP = false>
struct FwdLayout {
  static constexpr int ESZ = F8 ? 1 : 2;     // bytes per element
  static constexpr int QB = TILE * D * ESZ;  // one Q tile (bytes)
  static constexpr int TB = TILE * D * ESZ;  // one K or V tile
  static constexpr int STAGES = F8 ? 8 : (D == 64 ? 6 : 4);  // K/V tile slots
  // Slots are used in pairs: group 0 of a unit holds K_0, group j+1 holds V_j and
  // K_{j+1} (the two tiles the step after S_j reads), so a step costs the MMA
  // thread one wait and one release instead of two of each.
  static constexpr int NG = STAGES / 2;
  static constexpr int CH = D * ESZ / 128;   // 128-byte swizzle atoms per tile row
  static constexpr int ECH = 128 / ESZ;      // elements per atom row (the TMA box width)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * QB;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TB;
  // barriers: unit_full[2] unit_empty[2] q_full q_empty kv_full[NG] kv_empty[NG]
  //           s_full[2] p_full[2] o_full[2] o_empty[2] p_full2[2]
  //           list_full[2] (block-sparse)
  static constexpr int NBAR = 4 + 2 + 2 * NG + 10 + (SP ? 2 : 0);
  static constexpr int OFF_UNIT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_TMEM = OFF_UNIT + 16;
  static constexpr int OFF_SCR = (OFF_TMEM + 16 + 1023) / 1024 * 1024;  // output staging, one per softmax warp
  // two 2 KB boxes per warp for TMA stores (block-sparse: the row-store scratch)
  static constexpr int SCR = SP ? ROW_SCRATCH_BYTES : 4096;
  // block-sparse unit lists, one per unit slot: header (nu, n[2], first[2],
  // last[2]), per-key-tile flags of the two rows, then the union (act, kt)
  static constexpr int MAXL = 1024;  // key tiles (Nk <= 131072)
  static constexpr int LIST = SP ? (48 + 5 * MAXL + 127) / 128 * 128 : 0;
  static constexpr int OFF_LIST = OFF_SCR + 8 * SCR;
  static constexpr int BYTES = OFF_LIST + 2 * LIST;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory");
};

// A unit's key-tile list in shared memory (block-sparse).
struct SpList {
  int* hdr;       // [0] nu  [1..2] n[t]  [3..4] first step of t  [5..6] last step of t
  uint8_t* a0;    // key tile c listed for query tile 0 / 1 (build scratch)
  uint8_t* a1;
  uint8_t* act;   // union step j: bit t set when query tile t uses it
  int16_t* kt;    // union step j: key tile
};
template <int MAXL>
__device__ __forceinline__ SpList sp_list(uint8_t* base) {
  SpList l;
  l.hdr = reinterpret_cast<int*>(base);
  l.a0 = base + 48;
  l.a1 = l.a0 + MAXL;
  l.act = l.a1 + MAXL;
  l.kt = reinterpret_cast<int16_t*>(l.act + MAXL);
  return l;
}

struct FwdParams {
  Dims dims;
  float scale_log2;
  float tau;        // conditional rescaling threshold, log2 units (0: exact running max)
  const float* sq;  // FP8: Q block scales [B, Hq, nqt], K block scales [B, Hkv, nkt], V head scales [B, Hkv]
  const float* sk;
  const float* sv;
  int nqt, nkt;
  const int* row_ptr;  // block-sparse CSR table: [nqt + 1], col_idx [nnz]
  const int* col_idx;
  int nnz;
  const int* plan;     // packed sequences: the device-side work plan (units with work only)
  OutRows o;
  OutRows o_res;
  float* lse;
  int* status;
  int* counter;
  unsigned long long timeout_ns;
  int total_units;
  unsigned long long* trace;  // optional timestamps (see TRACE_UNIT0)
  int tma_out;                // O (and its residual) leave through TMA stores (dense)
  int split0, nsplit;         // key-split units: items from split0 on are parts (see FwdLaunch)
  float* part_o;
  float* part_lse;
};

struct Bars {
  uint64_t *unit_full, *unit_empty, *q_full, *q_empty, *kv_full, *kv_empty, *s_full, *p_full, *o_full, *o_empty;
  uint64_t* p_full2;    // [2]: the second half of a tile's P (keys 64-127; p_full: keys 0-63)
  uint64_t* list_full;  // block-sparse only
};

template <int D, bool F8, bool SP>
__device__ __forceinline__ Bars carve_bars(uint8_t* smem) {
  using L = FwdLayout<D, F8, SP>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  Bars r;
  r.unit_full = b;
  r.unit_empty = b + 2;
  r.q_full = b + 4;
  r.q_empty = b + 5;
  r.kv_full = b + 6;
  r.kv_empty = r.kv_full + L::NG;
  r.s_full = r.kv_empty + L::NG;
  r.p_full = r.s_full + 2;
  r.o_full = r.p_full + 2;
  r.o_empty = r.o_full + 2;
  r.list_full = r.o_empty + 2;
  r.p_full2 = r.list_full + (SP ? 2 : 0);
  return r;
}

// The key tiles of unit p: each query tile t visits [lo[t], hi[t]) (empty when
// the tile is past the sequence); the unit streams the union [base, base + nu)
// once, and tile t is active at local steps [a[t], a[t] + n[t]).
struct UnitTiles {
  int base, nu;
  int a[2], n[2];
};

// Without a band every range starts at key tile 0 and (under j <= i, where
// Nq == Nk) ends at the diagonal tile.
template <int MASK>
__device__ __forceinline__ UnitTiles unit_tiles(const Dims& s, int p) {
  const int nq = q_tiles(s);
  int lo[2], hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * p + t;
    lo[t] = hi[t] = 0;
    if (qt < nq) {
      if (MASK == MASK_BAND)
        kv_range(s, qt, lo[t], hi[t]);
      else
        hi[t] = MASK == MASK_CAUSAL ? qt + 1 : k_tiles(s);
    }
  }
  if (MASK != MASK_BAND) {
    UnitTiles u;
    u.base = 0;
    u.nu = imax(hi[0], hi[1]);
    u.a[0] = u.a[1] = 0;
    u.n[0] = hi[0];
    u.n[1] = hi[1];
    return u;
  }
  UnitTiles u;
  const bool e1 = hi[1] <= lo[1];  // tile 1 past the sequence (tile 0 never is)
  u.base = e1 ? lo[0] : imin(lo[0], lo[1]);
  u.nu = (e1 ? hi[0] : imax(hi[0], hi[1])) - u.base;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    u.n[t] = imax(0, hi[t] - lo[t]);
    u.a[t] = u.n[t] > 0 ? lo[t] - u.base : 0;
  }
  return u;
}

// A work unit's trace record (dense units; the index from (b, h, pair), so that no
// register has to keep it alive across the unit).
__device__ __forceinline__ unsigned long long* trace_unit(const FwdParams& p, int b, int h, int pr) {
  return p.trace + TRACE_UNIT0 + static_cast<int64_t>(fwd_unit_index(p.dims, b, h, pr)) * TRACE_UNIT_WORDS;
}

// The unit's (b, h, pair): dense order (a key-split part: its unit's), or the
// packed sequences' plan.
template <bool VL>
__device__ __forceinline__ void fwd_unit_of(const FwdParams& p, int u, int& b, int& h, int& pr) {
  if (VL)
    plan_unit(p.plan, p.dims.Hq, u, b, h, pr);
  else
    fwd_unit(p.dims, u < p.split0 ? u : p.split0 + (u - p.split0) / p.nsplit, b, h, pr);
}

// A key-split part (work item u >= split0 of an unmasked dense forward) streams
// only its share of the key tiles: part k of nsplit covers [k nk / nsplit,
// (k + 1) nk / nsplit) of the unit's nk.
template <int MASK, bool VL, bool SP>
__device__ __forceinline__ void split_tiles(const FwdParams& p, int u, UnitTiles& ut) {
  if (MASK != MASK_NONE || VL || SP || u < p.split0) return;
  const int k = (u - p.split0) % p.nsplit, nk = ut.nu;
  const int lo = k * nk / p.nsplit, hi = (k + 1) * nk / p.nsplit;
  ut.base = lo;
  ut.nu = hi - lo;
#pragma unroll
  for (int t = 0; t < 2; ++t) ut.n[t] = ut.n[t] > 0 ? hi - lo : 0;
}

template <bool VL>
__device__ __forceinline__ int fwd_total(const FwdParams& p) { return VL ? __ldg(p.plan) : p.total_units; }

// ------------------------------------------------------------------ producer
template <int D, int MASK, bool F8, bool VL, bool SP, int DG>
__device__ void fwd_producer(uint8_t* smem, const Bars& bar, int* unit_slot, const CUtensorMap* tm_q,
                             const CUtensorMap* tm_k, const CUtensorMap* tm_v, const FwdParams& p,
                             const FwdSched& sched, const Ctl& ctl) {
  using L = FwdLayout<D, F8, SP>;
  constexpr bool SKIP = VL || SP;  // units may have no work
  const int g = p.dims.Hq / p.dims.Hkv;
  uint32_t seq = 0;       // K/V groups issued so far (ring sequence number)
  uint32_t qn = 0;        // units with work so far (Q load phase)
  int q_armed = -1;       // phase of the last Q load issued
  const int total = fwd_total<VL>(p);
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!mbar_wait(&bar.unit_empty[slot], ((it >> 1) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
    int u;
    if (sched.on) {  // this CTA's list of the static schedule
      const int k = sched.start[blockIdx.x] + it;
      u = k < sched.start[blockIdx.x + 1] ? sched.ord[k] : total;
    } else {
      u = atomicAdd(p.counter, 1);
    }
    if (DG == DG_TRACE && u < total && u < p.split0) {  // (key-split parts are not traced)
      unsigned long long* rec = p.trace + TRACE_UNIT0 + static_cast<int64_t>(u) * TRACE_UNIT_WORDS;
      rec[0] = globaltimer();
      rec[3] = 0;
      rec[4] = blockIdx.x;
      p.trace[4 * blockIdx.x + 3] += 1;
    }
    unit_slot[slot] = u;
    mbar_arrive(&bar.unit_full[slot]);
    if (u >= total) break;
    int b, h, pr;
    fwd_unit_of<VL>(p, u, b, h, pr);
    const SeqRows sr = seq_rows<VL>(p.dims, b);
    UnitTiles ut = unit_tiles<MASK>(VL ? sr.s : p.dims, pr);
    split_tiles<MASK, VL, SP>(p, u, ut);
    int nmax = ut.nu;
    SpList sl{};
    if (SP) {  // the unit's key tiles, from the list warp 2 built
      if (!mbar_wait(&bar.list_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
      sl = sp_list<L::MAXL>(smem + L::OFF_LIST + slot * L::LIST);
      nmax = sl.hdr[0];
    }
    if (SKIP && nmax == 0) continue;  // no key tile for either query tile (past a packed sequence, or none listed)
    const int kvh = h / g;
    const int qrow = VL ? sr.qoff : 0, krow = VL ? sr.koff : 0, tb = VL ? 0 : b;
    auto key_tile = [&](int step) { return SP ? static_cast<int>(sl.kt[step]) : ut.base + step; };

    // The Q load must wait until the previous unit's last S has read the buffer;
    // bring the tiles into L2 now, so that the load then comes from L2.
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int c = 0; c < L::CH; ++c) tma_prefetch_l2_4d(tm_q, c * L::ECH, h, qrow + (2 * pr + t) * TILE, tb);
    if (!mbar_wait(bar.q_empty, ((SKIP ? qn : it) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) break;
    mbar_arrive_expect_tx(bar.q_full, 2 * L::QB);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int c = 0; c < L::CH; ++c)
        tma_load_4d(smem + L::OFF_Q + t * L::QB + c * (TILE * 128), tm_q, bar.q_full, c * L::ECH, h,
                    qrow + (2 * pr + t) * TILE, tb);
    q_armed = SKIP ? static_cast<int>(qn++) : it;

    bool ok = true;
    for (int gi = 0; gi <= nmax; ++gi, ++seq) {  // group gi: V_{gi-1} (slot A), K_gi (slot B)
      const int gs = seq % L::NG;
      if (!mbar_wait(&bar.kv_empty[gs], ((seq / L::NG) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) {
        ok = false;
        break;
      }
      const bool has_v = gi > 0, has_k = gi < nmax;
      uint8_t* base = smem + L::OFF_KV + gs * 2 * L::TB;
      mbar_arrive_expect_tx(&bar.kv_full[gs], (has_v + has_k) * L::TB);
#pragma unroll
      for (int c = 0; c < L::CH; ++c) {
        if (has_v)
          tma_load_4d(base + c * (TILE * 128), tm_v, &bar.kv_full[gs], c * L::ECH, kvh,
                      krow + key_tile(gi - 1) * TILE, tb);
        if (has_k)
          tma_load_4d(base + L::TB + c * (TILE * 128), tm_k, &bar.kv_full[gs], c * L::ECH, kvh,
                      krow + key_tile(gi) * TILE, tb);
      }
    }
    if (!ok) break;
  }
  // Let every copy still in flight land before the CTA can exit.
  for (int gs = 0; gs < L::NG; ++gs) {
    if (seq > static_cast<uint32_t>(gs)) {
      const uint32_t last = seq - 1 - ((seq - 1 - gs) % L::NG);  // last group issued on slot pair gs
      mbar_wait(&bar.kv_full[gs], (last / L::NG) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
    }
  }
  if (q_armed >= 0) mbar_wait(bar.q_full, q_armed & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
}

// ------------------------------------------------------------------ MMA issuer
// Run by the whole warp, converged: every wait is the warp's, and one elected
// lane issues each MMA and commit, so the descriptors are formed once per warp in
// uniform registers (a single diverged lane forming them issues far slower).
template <int D, int MASK, bool F8, bool VL, bool SP, int DG>
__device__ void fwd_mma(uint8_t* smem, const Bars& bar, const int* unit_slot, uint32_t tmem, const FwdParams& p,
                        const Ctl& ctl) {
  using L = FwdLayout<D, F8, SP>;
  constexpr bool SKIP = VL || SP;
  // Q K^T with both operands K-major; P V with V N-major
  constexpr uint32_t IDESC_S = F8 ? idesc_e4m3(128, 128, false, false) : idesc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_O = F8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
  constexpr int KS = F8 ? 32 : 16;  // K of one product (32 bytes of a 128-byte swizzle row)
  const uint32_t q_base = smem_u32(smem + L::OFF_Q);
  const uint32_t kv_base = smem_u32(smem + L::OFF_KV);
  uint32_t seq = 0;
  uint32_t qn = 0;  // units with work so far (Q phase)
  uint32_t pph[2] = {0, 0};
  uint32_t active[2] = {0, 0};

  auto issue_s = [&](int t, uint32_t k_addr) {
    const uint32_t d_tmem = tmem + t * 128;
#pragma unroll
    for (int k = 0; k < D / KS; ++k) {
      const uint32_t off = (k / 4) * (TILE * 128) + (k % 4) * 32;
      const uint64_t a = sdesc_sw128(q_base + t * L::QB + off, 16, 1024);
      const uint64_t bd = sdesc_sw128(k_addr + off, 16, 1024);
      if (elect_one()) {
        if (F8)
          mma_ss_f8(d_tmem, a, bd, IDESC_S, k > 0);
        else
          mma_ss(d_tmem, a, bd, IDESC_S, k > 0);
      }
    }
  };
  // P is read from TMEM, 8 columns per product (8 x 2 bf16 or 8 x 4 E4M3 keys)
  auto issue_pv = [&](int t, uint32_t v_addr, bool acc, int half) {  // half: the keys 64 h .. 64 h + 63
    const uint32_t d_tmem = tmem + 256 + t * D;
    const uint32_t p_tmem = tmem + t * 128;
#pragma unroll
    for (int k = half * (TILE / KS / 2); k < (half + 1) * (TILE / KS / 2); ++k) {
      const uint64_t bd = sdesc_sw128(v_addr + k * KS * 128, TILE * 128, 1024);
      if (elect_one()) {
        if (F8)
          mma_ts_f8(d_tmem, p_tmem + k * 8, bd, IDESC_O, (acc || k > 0) ? 1u : 0u);
        else
          mma_ts(d_tmem, p_tmem + k * 8, bd, IDESC_O, (acc || k > 0) ? 1u : 0u);
      }
    }
  };
  auto group_wait = [&](uint32_t gq) {
    return warp_wait(&bar.kv_full[gq % L::NG], (gq / L::NG) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
  };
  auto group_base = [&](uint32_t gq) { return kv_base + (gq % L::NG) * 2 * L::TB; };

  const int total = fwd_total<VL>(p);
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!warp_wait(&bar.unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT)) return;
    const int u = unit_slot[slot];
    if ((!SP || u >= total) && elect_one()) mbar_arrive(&bar.unit_empty[slot]);  // block-sparse: after the unit
    if (u >= total) return;
    int b, h, pr;
    fwd_unit_of<VL>(p, u, b, h, pr);
    UnitTiles ut = unit_tiles<MASK>(VL ? seq_rows<VL>(p.dims, b).s : p.dims, pr);
    split_tiles<MASK, VL, SP>(p, u, ut);
    int nmax = ut.nu;
    // tile t is active at local steps [a[t], e[t]) (block-sparse: the steps its bit marks)
    int a[2] = {ut.a[0], ut.a[1]}, e[2] = {ut.a[0] + ut.n[0], ut.a[1] + ut.n[1]}, nt[2] = {ut.n[0], ut.n[1]};
    SpList sl{};
    if (SP) {
      if (!warp_wait(&bar.list_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_MMA)) return;
      sl = sp_list<L::MAXL>(smem + L::OFF_LIST + slot * L::LIST);
      nmax = sl.hdr[0];
      for (int t = 0; t < 2; ++t) {
        nt[t] = sl.hdr[1 + t];
        a[t] = sl.hdr[3 + t];
        e[t] = sl.hdr[5 + t] + 1;
      }
    }
    auto on = [&](int t, int j) { return SP ? ((sl.act[j] >> t) & 1) != 0 : (j >= a[t] && j < e[t]); };
    if (SKIP && nmax == 0) {  // no key tile for either query tile
      if (SP && elect_one()) mbar_arrive(&bar.unit_empty[slot]);
      continue;
    }

    if (!warp_wait(bar.q_full, (SKIP ? qn++ : static_cast<uint32_t>(it)) & 1, ctl, FA_STATUS_TIMEOUT_MMA)) return;
    unsigned long long* rec =
        DG == DG_TRACE && u < p.split0 ? p.trace + TRACE_UNIT0 + static_cast<int64_t>(u) * TRACE_UNIT_WORDS : nullptr;
    // group 0: K of local step 0
    {
      if (!group_wait(seq)) return;
      if (rec && lane_id() == 0) rec[1] = globaltimer();
      tc_fence_after();
      for (int t = 0; t < 2; ++t)
        if (nt[t] > 0 && on(t, 0)) {
          issue_s(t, group_base(seq) + L::TB);
          if (elect_one()) mma_commit(&bar.s_full[t]);
        }
      if (elect_one()) {
        if (nmax == 1) mma_commit(bar.q_empty);
        mma_commit(&bar.kv_empty[seq % L::NG]);
      }
    }
    for (int j = 0; j < nmax; ++j) {
      const uint32_t gq = seq + 1 + j;  // group j+1: V_j, and K_{j+1} unless this is the last step
      if (!group_wait(gq)) return;
      const uint32_t v_addr = group_base(gq), k_addr = v_addr + L::TB;
      for (int t = 0; t < 2; ++t) {
        const bool now = on(t, j);
        if (now) {
          if (j == a[t] && !warp_wait(&bar.o_empty[t], (active[t] & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_MMA)) return;
          // P V in two halves of the keys, each as soon as its half of P is in TMEM
          // (E4M3: one hand-off; half a P V is two products, too short to overlap)
          if (!warp_wait(&bar.p_full[t], pph[t], ctl, FA_STATUS_TIMEOUT_MMA)) return;
          tc_fence_after();
          issue_pv(t, v_addr, j > a[t], 0);
          if (!F8) {
            if (!warp_wait(&bar.p_full2[t], pph[t], ctl, FA_STATUS_TIMEOUT_MMA)) return;
            tc_fence_after();
          }
          pph[t] ^= 1;
          issue_pv(t, v_addr, true, 1);
          if (j == e[t] - 1 && elect_one()) mma_commit(&bar.o_full[t]);
        }
        if (j + 1 < nmax && on(t, j + 1)) {  // S of the tile's next step (its first, when it starts late)
          if (!now) tc_fence_after();         // no P V of this tile in this step fenced the group wait
          issue_s(t, k_addr);
          if (elect_one()) mma_commit(&bar.s_full[t]);
        }
      }
      if (elect_one()) {
        if (j + 1 == nmax - 1) mma_commit(bar.q_empty);
        mma_commit(&bar.kv_empty[gq % L::NG]);
      }
    }
    if (rec && lane_id() == 0) rec[2] = globaltimer();
    for (int t = 0; t < 2; ++t)
      if (nt[t] > 0) ++active[t];
    seq += nmax + 1;
    if (SP && elect_one()) mbar_arrive(&bar.unit_empty[slot]);
  }
}

// One warp's 32 rows x 32 bf16 columns (w: this lane's row, packed in pairs) leave
// through a TMA store of a 64-byte-swizzled box staged in `buf` (2 KB, 512-byte
// aligned): 16-byte chunk q of row r sits at chunk q ^ ((r / 2) % 4).  Rows past the
// tensor's end are dropped by the copy engine.  Each warp alternates two buffers;
// before one is refilled, the store made from it two boxes ago must have read it
// (at most one group, the previous box's, may still be reading).
__device__ __forceinline__ void stage_box_store(const uint32_t (&w)[16], uint8_t* buf, const CUtensorMap* map,
                                                int c0, int c1, int c2, int c3) {
  const int lr = lane_id();
  if (lr == 0) bulk_wait_read<1>();
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(buf + lr * 64 + ((q ^ ((lr >> 1) & 3)) << 4)) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lr == 0) {
    tma_store_4d(map, buf, c0, c1, c2, c3);
    bulk_commit();
  }
}

// ------------------------------------------------------------------ softmax
template <int D, int MASK, bool F8, bool VL, bool SP, int DG>
__device__ void fwd_softmax(int t, uint8_t* smem, const Bars& bar, const int* unit_slot, uint32_t tmem,
                            const FwdParams& p, const Ctl& ctl, uint8_t* scratch, const CUtensorMap* tm_o,
                            const CUtensorMap* tm_r) {
  using L = FwdLayout<D, F8, SP>;
  const int wq = (threadIdx.x >> 5) & 3;  // warp within the warpgroup = TMEM lane quarter
  const int r = wq * 32 + lane_id();      // row of the query tile
  const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lanes + t * 128;
  const uint32_t tO = tmem + lanes + 256 + t * D;
  const float c = p.scale_log2;
  const Dims& s = p.dims;
  uint32_t sph = 0, active = 0;
  uint32_t nbox = 0;  // output boxes staged so far (TMA stores alternate two buffers)
  const int total = fwd_total<VL>(p);

  for (int it = 0;; ++it) {
    const int slot = it & 1;
    bool ok = mbar_wait(&bar.unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT);
    if (!__all_sync(0xffffffffu, ok)) return;
    const int u = unit_slot[slot];
    if (!SP || u >= total) warp_arrive(&bar.unit_empty[slot]);  // block-sparse: after the unit
    if (u >= total) return;
    int b, h, pr;
    fwd_unit_of<VL>(p, u, b, h, pr);
    const SeqRows sr = seq_rows<VL>(s, b);
    if (VL && !sr.ok && t == 0 && wq == 0 && lane_id() == 0) report(ctl, FA_STATUS_BAD_INPUT);
    const Dims& su = VL ? sr.s : s;  // this unit's sequence (packed), else the problem
    UnitTiles ut = unit_tiles<MASK>(su, pr);
    split_tiles<MASK, VL, SP>(p, u, ut);
    const bool part = MASK == MASK_NONE && !VL && !SP && u >= p.split0;  // a key-split part
    int n = ut.n[t];
    const int qt = 2 * pr + t;
    SpList sl{};
    if (SP) {
      ok = mbar_wait(&bar.list_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT);
      if (!__all_sync(0xffffffffu, ok)) return;
      sl = sp_list<L::MAXL>(smem + L::OFF_LIST + slot * L::LIST);
      n = sl.hdr[1 + t];
      if (n == 0 && qt < q_tiles(s)) {  // no key tile listed: O = 0, LSE = -inf
        const int q0 = qt * TILE + wq * 32;
        __nv_bfloat16* o0 = reinterpret_cast<__nv_bfloat16*>(p.o.ptr) + b * p.o.sb +
                            static_cast<int64_t>(q0) * p.o.sn + h * p.o.sh;
        uint32_t zw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) zw[i] = 0u;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) store_rows32_bf16(zw, scratch, o0 + cc * 32, p.o.sn, s.Nq - q0);
        if (p.o_res.ptr != nullptr) {
          __nv_bfloat16* r0 = reinterpret_cast<__nv_bfloat16*>(p.o_res.ptr) + b * p.o_res.sb +
                              static_cast<int64_t>(q0) * p.o_res.sn + h * p.o_res.sh;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) store_rows32_bf16(zw, scratch, r0 + cc * 32, p.o_res.sn, s.Nq - q0);
        }
        if (qt * TILE + r < s.Nq) p.lse[(static_cast<int64_t>(b) * s.Hq + h) * s.Nq + qt * TILE + r] = -INFINITY;
      }
      if (n == 0) warp_arrive(&bar.unit_empty[slot]);
    }
    if (n == 0) continue;
    const int nq_u = su.Nq, nk_u = su.Nk, qoff = VL ? sr.qoff : 0;
    const int q_row = qt * TILE + r;
    int jj = 0;  // block-sparse: scan position in the unit's list
    const int kt0 = ut.base + ut.a[t];  // first key tile of this query tile
    // FP8: logits = S * scale*log2(e) * s_q * s_k[kt]; a zero block scale leaves S = 0
    // exactly, and the floor keeps masked -inf scores from becoming NaN
    const int kvh = h / (s.Hq / s.Hkv);
    const float cq = F8 ? c * p.sq[(static_cast<int64_t>(b) * s.Hq + h) * p.nqt + qt] : c;
    const float* skp = F8 ? p.sk + (static_cast<int64_t>(b) * s.Hkv + kvh) * p.nkt + kt0 : nullptr;
    int full_lo = 0, full_hi = 0;        // band: key tiles this query tile sees in full
    if (MASK == MASK_BAND) {
      kv_full_range(su, qt, full_lo, full_hi);
      if ((nk_u % TILE) != 0) full_hi = imin(full_hi, cdiv(nk_u, TILE) - 2);  // the ragged last tile is masked too
    }

    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < n; ++j) {
      const float cj = F8 ? fmaxf(cq * __ldg(skp + j), 1.17549435e-38f) : c;
      const float2 cj2 = make_float2(cj, cj);
      ok = mbar_wait(&bar.s_full[t], sph, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
      sph ^= 1;
      if (!__all_sync(0xffffffffu, ok)) return;
      if (DG == DG_TRACE && j == 0 && wq == 0 && lane_id() == 0) trace_unit(p, b, h, pr)[5 + t] = globaltimer();
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld128(tS, sr);

      float sv[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sv[i] = __uint_as_float(sr[i]);
      if (SP) {  // this step's key tile: the next list entry marked for this query tile
        while (((sl.act[jj] >> t) & 1) == 0) ++jj;
        const int kt = sl.kt[jj++];
        if ((MASK == MASK_CAUSAL && kt == qt) || (kt == k_tiles(s) - 1 && (nk_u % TILE) != 0)) {
          int lim = nk_u - kt * TILE;  // keys at or past Nk, and under j <= i keys past the row
          if (MASK == MASK_CAUSAL) lim = imin(lim, q_row - kt * TILE + 1);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) sv[i] = -INFINITY;
        }
      } else if (MASK == MASK_BAND) {
        const int kt = kt0 + j;
        if (kt < full_lo || kt > full_hi) {
          // keys [lo, hi) of this tile are visible to the row: the band i - wl .. i + wr, below Nk
          const int hi = imin(nk_u - kt * TILE, imin(TILE, q_row + s.wr + 1 - kt * TILE));
          const int lo = imax(0, q_row - s.wl - kt * TILE);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= hi || i < lo) sv[i] = -INFINITY;
        }
      } else if (MASK == MASK_CAUSAL ? j == n - 1 : ((nk_u % TILE) != 0 && kt0 + j == cdiv(nk_u, TILE) - 1)) {
        // the last tile: keys at or past Nk, and under j <= i keys past the row (a
        // key-split part starts at key tile kt0 and holds the last tile only if it ends there)
        int lim = nk_u - (kt0 + j) * TILE;
        if (MASK == MASK_CAUSAL) lim = imin(lim, q_row - j * TILE + 1);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) sv[i] = -INFINITY;
      }
      // Row max (three-input max), then exp2 and row sum on packed f32x2 operations:
      // scalar FP32 issue at this rate from several sub-partitions slows the tensor pipe.
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; i += 8) {
        mx0 = fmax3(mx0, sv[i], sv[i + 1]);
        mx1 = fmax3(mx1, sv[i + 2], sv[i + 3]);
        mx2 = fmax3(mx2, sv[i + 4], sv[i + 5]);
        mx3 = fmax3(mx3, sv[i + 6], sv[i + 7]);
      }
      const float m_tile = fmaxf(fmax3(mx0, mx1, mx2), mx3) * cj;
      const float m_new = (m_tile > m_run + p.tau) ? m_tile : m_run;
      // Under a band a row may see no key of a tile: while it has seen none at all, m
      // stays -inf, alpha 1 and every p 0.  (Causal and full rows see a key in their
      // first tile.  Measured: the guarded form costs the causal kernels 1-2% and saves
      // the full d = 64 kernel 5%, hence the split.)
      const float alpha = (MASK == MASK_CAUSAL) ? ex2(m_run - m_new) : (m_new == m_run) ? 1.f : ex2(m_run - m_new);
      const float m_use = (MASK == MASK_BAND && m_new == -INFINITY) ? 0.f : m_new;
      // FP8: p' = 448 p / 2^tau (P <= 2^tau fixes P's scale at 2^tau / 448), and l sums p' alike
      const float off = F8 ? (LOG2_448 - p.tau) - m_use : -m_use;
      const float2 neg_m2 = make_float2(off, off);
      float2 sum0 = make_float2(0.f, 0.f), sum1 = make_float2(0.f, 0.f);
      uint32_t pk[64];
      // P in two halves of the keys: the first half's P V starts while the second
      // half's exponentials run (E4M3: one store of all 128 keys, both halves at once)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int i = 32 * hf; i < 32 * hf + 32; i += 2) {
          const float2 x0 = __ffma2_rn(make_float2(sv[2 * i], sv[2 * i + 1]), cj2, neg_m2);
          const float2 x1 = __ffma2_rn(make_float2(sv[2 * i + 2], sv[2 * i + 3]), cj2, neg_m2);
          const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
          const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
          sum0 = __fadd2_rn(sum0, p0);
          sum1 = __fadd2_rn(sum1, p1);
          if (F8) {
            pk[i >> 1] = pack4_e4m3(p0.x, p0.y, p1.x, p1.y);
          } else {
            pk[i] = pack_bf16(p0.x, p0.y);
            pk[i + 1] = pack_bf16(p1.x, p1.y);
          }
        }
        if (F8 && hf == 0) continue;
        if (F8)
          tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        else
          tmem_st32(tS + 32 * hf, *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * hf]));
        if (hf == 0 && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // O *= alpha before its P V
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v = __fmul2_rn(f32x2(o[2 * i], o[2 * i + 1]), a2);
              o[2 * i] = __float_as_uint(v.x);
              o[2 * i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + cc * 32, o);
          }
        }
        if (F8 && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v = __fmul2_rn(f32x2(o[2 * i], o[2 * i + 1]), a2);
              o[2 * i] = __float_as_uint(v.x);
              o[2 * i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + cc * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        if (hf == 0 || F8) {
          // (test instantiation: the first warp of query tile 0 of work unit 0 withholds its first hand-off)
          if (DG != DG_WITHHOLD || u != 0 || j != 0 || t != 0 || wq != 0) warp_arrive(&bar.p_full[t]);
        }
        if (hf == 1 && !F8) warp_arrive(&bar.p_full2[t]);
      }
      l_run = l_run * alpha + ((sum0.x + sum0.y) + (sum1.x + sum1.y));
      if (DG == DG_TRACE && j == n - 1 && wq == 0 && lane_id() == 0) trace_unit(p, b, h, pr)[7 + t] = globaltimer();
      m_run = m_new;
    }

    // epilogue: O / l -> bf16, LSE
    ok = mbar_wait(&bar.o_full[t], active & 1, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
    ++active;
    if (!__all_sync(0xffffffffu, ok)) return;
    if (DG == DG_TRACE && wq == 0 && lane_id() == 0) trace_unit(p, b, h, pr)[9 + t] = globaltimer();
    tc_fence_after();
    const float inv_l = (F8 ? p.sv[static_cast<int64_t>(b) * s.Hkv + kvh] : 1.f) / l_run;
    const float2 il2 = make_float2(inv_l, inv_l);
    if (part) {  // a key-split part: its O / l (fp32) and LSE go to the workspace for the combine
      const int64_t prow = (static_cast<int64_t>(u - p.split0) * 2 + t) * TILE + r;
      float4* po = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 a = __fmul2_rn(f32x2(o[4 * i], o[4 * i + 1]), il2);
          const float2 c2 = __fmul2_rn(f32x2(o[4 * i + 2], o[4 * i + 3]), il2);
          po[cc * 8 + i] = make_float4(a.x, a.y, c2.x, c2.y);
        }
      }
      p.part_lse[prow] = (m_run + __log2f(l_run)) * LN2;
      tc_fence_before();
      warp_arrive(&bar.o_empty[t]);
      continue;
    }
    const bool live = q_row < nq_u;
    const int q0 = qt * TILE + wq * 32;  // this warp's first row (within its sequence)
    const int64_t orow = qoff + q0;      // ... and in the tensor
    __nv_bfloat16* o0 = reinterpret_cast<__nv_bfloat16*>(p.o.ptr) + b * p.o.sb + orow * p.o.sn + h * p.o.sh;
    __nv_bfloat16* r0 = p.o_res.ptr == nullptr ? nullptr
                                               : reinterpret_cast<__nv_bfloat16*>(p.o_res.ptr) + b * p.o_res.sb +
                                                     orow * p.o_res.sn + h * p.o_res.sh;
    // Kept rolled: the epilogue runs once per unit, so its code is cold in the SM's
    // instruction cache more often than not, and a quarter of it is a quarter of the
    // fetches (measured: with another kernel's code in between launches, the causal
    // N4096 forward 0.1298 -> 0.1254 ms; unchanged when the code stays cached).
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o[32];
      tmem_ld32(tO + cc * 32, o);

      float2 ov[16];
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ov[i] = __fmul2_rn(f32x2(o[2 * i], o[2 * i + 1]), il2);
        w[i] = pack_bf16(ov[i].x, ov[i].y);
      }
      if (!VL && !SP && p.tma_out) {  // TMA stores: this warp's 32 rows x 32 channels as one box
        if (q0 >= nq_u) continue;     // every row of this warp lies past the end
        stage_box_store(w, scratch + (nbox++ & 1) * 2048, tm_o, cc * 32, h, q0, b);
        if (p.o_res.ptr != nullptr) {  // rounding residual: bf16(O - bf16(O))
          uint32_t rz[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 hv = unpack_bf16(w[i]);
            rz[i] = pack_bf16(ov[i].x - hv.x, ov[i].y - hv.y);
          }
          stage_box_store(rz, scratch + (nbox++ & 1) * 2048, tm_r, cc * 32, h, q0, b);
        }
        continue;
      }
      store_rows32_bf16(w, scratch, o0 + cc * 32, p.o.sn, nq_u - q0);
      if (r0 != nullptr) {  // rounding residual: bf16(O - bf16(O))
        uint32_t rz[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 hv = unpack_bf16(w[i]);
          rz[i] = pack_bf16(ov[i].x - hv.x, ov[i].y - hv.y);
        }
        store_rows32_bf16(rz, scratch, r0 + cc * 32, p.o_res.sn, nq_u - q0);
      }
    }
    if (live)  // LSE [B, Hq, Nq], or [Hq, total_q] for packed sequences
      p.lse[(VL ? static_cast<int64_t>(h) * s.total_q + qoff : (static_cast<int64_t>(b) * s.Hq + h) * s.Nq) +
            q_row] = (m_run + __log2f(l_run) - (F8 ? LOG2_448 - p.tau : 0.f)) * LN2;
    tc_fence_before();
    warp_arrive(&bar.o_empty[t]);
    if (DG == DG_TRACE && wq == 0 && lane_id() == 0) {
      unsigned long long* rec = trace_unit(p, b, h, pr);
      const unsigned long long now = globaltimer();
      rec[11 + t] = now;
      atomicMax(rec + 3, now);
    }
    if (SP) warp_arrive(&bar.unit_empty[slot]);
  }
}

// ------------------------------------------------------------------ block-sparse lists (warp 2)
// For each unit: mark the key tiles each of its two query tiles lists (entries
// must increase strictly within a row and lie below k_tiles; others are skipped
// and reported; under j <= i tiles above the diagonal hide every key and are
// skipped), then compact the marks into the union in key order.
template <int D, int MASK>
__device__ void fwd_sparse_lists(uint8_t* smem, const Bars& bar, const int* unit_slot, const FwdParams& p,
                                 const Ctl& ctl) {
  using L = FwdLayout<D, false, true>;
  const int lane = lane_id();
  const Dims& s = p.dims;
  const int nqt = q_tiles(s), nkt = k_tiles(s);
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    const bool ok = mbar_wait(&bar.unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT);
    if (!__all_sync(0xffffffffu, ok)) return;
    const int u = unit_slot[slot];
    warp_arrive(&bar.unit_empty[slot]);
    if (u >= p.total_units) return;
    int b, h, pr;
    fwd_unit(s, u, b, h, pr);
    const SpList sl = sp_list<L::MAXL>(smem + L::OFF_LIST + slot * L::LIST);
    for (int c = lane; c < nkt; c += 32) {
      sl.a0[c] = 0;
      sl.a1[c] = 0;
    }
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int qt = 2 * pr + t;
      if (qt >= nqt) continue;
      const int e0 = __ldg(p.row_ptr + qt), e1 = __ldg(p.row_ptr + qt + 1);
      if (e0 < 0 || e1 < e0 || e1 > p.nnz) {
        bad = true;
        continue;
      }
      uint8_t* mark = t ? sl.a1 : sl.a0;
      for (int e = e0 + lane; e < e1; e += 32) {
        const int c = __ldg(p.col_idx + e);
        const int prev = e > e0 ? __ldg(p.col_idx + e - 1) : -1;
        if (c <= prev || c < 0 || c >= nkt) {
          bad = true;
          continue;
        }
        if (MASK == MASK_CAUSAL && c > qt) continue;
        mark[c] = 1;
      }
    }
    __syncwarp();
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(ctl, FA_STATUS_BAD_INPUT);
    int nu = 0, n0 = 0, n1 = 0, f0 = -1, f1 = -1, l0 = -1, l1 = -1;
    for (int base = 0; base < nkt; base += 32) {
      const int c = base + lane;
      const int x0 = c < nkt ? sl.a0[c] : 0, x1 = c < nkt ? sl.a1[c] : 0;
      const unsigned m = __ballot_sync(0xffffffffu, x0 | x1);
      const unsigned m0 = __ballot_sync(0xffffffffu, x0), m1 = __ballot_sync(0xffffffffu, x1);
      const unsigned below = (1u << lane) - 1u;
      if (x0 | x1) {
        const int pos = nu + __popc(m & below);
        sl.kt[pos] = static_cast<int16_t>(c);
        sl.act[pos] = static_cast<uint8_t>(x0 | (x1 << 1));
      }
      // union positions of each query tile's first and last key tile
      if (m0) {
        if (f0 < 0) f0 = nu + __popc(m & ((1u << (__ffs(m0) - 1)) - 1u));
        l0 = nu + __popc(m & ((1u << (31 - __clz(m0))) - 1u));
      }
      if (m1) {
        if (f1 < 0) f1 = nu + __popc(m & ((1u << (__ffs(m1) - 1)) - 1u));
        l1 = nu + __popc(m & ((1u << (31 - __clz(m1))) - 1u));
      }
      nu += __popc(m);
      n0 += __popc(m0);
      n1 += __popc(m1);
    }
    if (lane == 0) {
      sl.hdr[0] = nu;
      sl.hdr[1] = n0;
      sl.hdr[2] = n1;
      sl.hdr[3] = f0;
      sl.hdr[4] = f1;
      sl.hdr[5] = l0;
      sl.hdr[6] = l1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.list_full[slot]);
  }
}

template <int D, int MASK, bool F8, bool VL, bool SP, int DG>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p,
                  const __grid_constant__ FwdSched sched, const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ CUtensorMap tm_r) {
  using L = FwdLayout<D, F8, SP>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Bars bar = carve_bars<D, F8, SP>(smem);
  int* unit_slot = reinterpret_cast<int*>(smem + L::OFF_UNIT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const Ctl ctl{p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(&bar.unit_full[0], 1);
    mbar_init(&bar.unit_full[1], 1);
    mbar_init(&bar.unit_empty[0], 1 + 8 + (SP ? 1 : 0));  // MMA, softmax warps (, list warp)
    mbar_init(&bar.unit_empty[1], 1 + 8 + (SP ? 1 : 0));
    if (SP) {
      mbar_init(&bar.list_full[0], 1);
      mbar_init(&bar.list_full[1], 1);
    }
    mbar_init(bar.q_full, 1);
    mbar_init(bar.q_empty, 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&bar.kv_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.p_full[t], 4);
      mbar_init(&bar.p_full2[t], 4);
      mbar_init(&bar.o_full[t], 1);
      mbar_init(&bar.o_empty[t], 4);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above touches only this CTA's own memory; from here on the kernel
  // reads the workspace header the previous kernel cleared, and the inputs
  griddep_wait();
  // a kernel queued behind this one with programmatic serialisation (the key-split
  // combine) may be scheduled now; it waits for this grid's completion itself
  griddep_launch_dependents();
  if (DG == DG_TRACE) {
    if (threadIdx.x == 0) {
      p.trace[4 * blockIdx.x] = globaltimer();
      p.trace[4 * blockIdx.x + 1] = 0;
      p.trace[4 * blockIdx.x + 2] = smid();
      p.trace[4 * blockIdx.x + 3] = 0;
    }
    __syncthreads();
  }

  if (warp == 0) {
    if (lane_id() == 0) fwd_producer<D, MASK, F8, VL, SP, DG>(smem, bar, unit_slot, &tm_q, &tm_k, &tm_v, p, sched, ctl);
  } else if (warp == 1) {
    fwd_mma<D, MASK, F8, VL, SP, DG>(smem, bar, unit_slot, tmem, p, ctl);
  } else if (SP && warp == 2) {
    fwd_sparse_lists<D, MASK>(smem, bar, unit_slot, p, ctl);
  } else if (warp >= 4) {
    fwd_softmax<D, MASK, F8, VL, SP, DG>((warp - 4) >> 2, smem, bar, unit_slot, tmem, p, ctl,
                                         smem + L::OFF_SCR + (warp - 4) * L::SCR, &tm_o, &tm_r);
    if (!VL && !SP && p.tma_out && lane_id() == 0) bulk_wait<0>();  // the output stores have finished
  }
  // the CTA's end: the last role to finish (each warp's lane 0 stamps its exit)
  if (DG == DG_TRACE && lane_id() == 0) atomicMax(p.trace + 4 * blockIdx.x + 1, globaltimer());
  // Lanes 1-31 of the producer warp had no role: they wait here for their lane 0,
  // so that every warp reaches the block barrier converged (the barrier is the
  // aligned form, which assumes whole warps) and TMEM is freed after all its users.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ key-split combine
// The nsplit parts' LSE-weighted sum (each part's O is normalised by its own sum),
// as the decode path combines its splits: LSE = log sum_k e^{LSE_k},
// O = sum_k e^{LSE_k - LSE} O_k.  A thread takes 8 columns of one row, so its
// loads (every part's LSE and columns) are all in flight at once.  Writes O
// (bf16), its rounding residual when asked for, and LSE.  Launched right behind
// the forward with programmatic serialisation: it waits for the forward's results.
template <int D>
__global__ void __launch_bounds__(128) fwd_split_combine_kernel(const FwdParams p) {
  constexpr int CPR = D / 8, RPB = 128 / CPR;  // 8-column chunks per row, rows per block
  griddep_wait();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / CPR;  // (unit, tile, row) of the splits
  const int c = (threadIdx.x % CPR) * 8;
  const int su = static_cast<int>(g / (2 * TILE)), t = static_cast<int>((g / TILE) & 1), r = static_cast<int>(g % TILE);
  int b, h, pr;
  fwd_unit(p.dims, p.split0 + su, b, h, pr);
  const int row = (2 * pr + t) * TILE + r;
  if (row >= p.dims.Nq) return;
  const int ns = p.nsplit;
  float l[4], w[4];
  float4 x0[4], x1[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // nsplit <= 4
    if (k < ns) {
      const int64_t pr_k = (static_cast<int64_t>(su * ns + k) * 2 + t) * TILE + r;
      l[k] = p.part_lse[pr_k];
      const float4* src = reinterpret_cast<const float4*>(p.part_o + pr_k * D + c);
      x0[k] = src[0];
      x1[k] = src[1];
    }
  }
  float mx = l[0];
#pragma unroll
  for (int k = 1; k < 4; ++k)
    if (k < ns) mx = fmaxf(mx, l[k]);
  float wsum = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < ns) {
      w[k] = expf(l[k] - mx);
      wsum += w[k];
      acc[0] += w[k] * x0[k].x;
      acc[1] += w[k] * x0[k].y;
      acc[2] += w[k] * x0[k].z;
      acc[3] += w[k] * x0[k].w;
      acc[4] += w[k] * x1[k].x;
      acc[5] += w[k] * x1[k].y;
      acc[6] += w[k] * x1[k].z;
      acc[7] += w[k] * x1[k].w;
    }
  }
  const float inv = 1.f / wsum;
  uint32_t ob[4], rb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float v0 = acc[2 * i] * inv, v1 = acc[2 * i + 1] * inv;
    ob[i] = pack_bf16(v0, v1);
    const float2 hv = unpack_bf16(ob[i]);
    rb[i] = pack_bf16(v0 - hv.x, v1 - hv.y);
  }
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.o.ptr) + b * p.o.sb + static_cast<int64_t>(row) * p.o.sn +
                     h * p.o.sh + c;
  *reinterpret_cast<uint4*>(o) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  if (p.o_res.ptr != nullptr) {
    __nv_bfloat16* res = reinterpret_cast<__nv_bfloat16*>(p.o_res.ptr) + b * p.o_res.sb +
                         static_cast<int64_t>(row) * p.o_res.sn + h * p.o_res.sh + c;
    *reinterpret_cast<uint4*>(res) = make_uint4(rb[0], rb[1], rb[2], rb[3]);
  }
  if (c == 0) p.lse[(static_cast<int64_t>(b) * p.dims.Hq + h) * p.dims.Nq + row] = mx + logf(wsum);
}

template <int D, int MASK, bool F8 = false, bool VL = false, bool SP = false, int DG = DG_NONE>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t st) {
  using L = FwdLayout<D, F8, SP>;
  auto kern = fa_fwd_kernel<D, MASK, F8, VL, SP, DG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.dims = a.dims;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.tau = a.tau;
  p.tma_out = (!VL && !SP) ? a.tma_out : 0;
  p.sq = a.sq;
  p.sk = a.sk;
  p.sv = a.sv;
  p.nqt = q_tiles(a.dims);
  p.nkt = k_tiles(a.dims);
  p.row_ptr = a.row_ptr;
  p.col_idx = a.col_idx;
  p.nnz = a.nnz;
  p.plan = a.plan;
  if (VL) {  // the units with work, longest first
    e = launch_varlen_plan(a.dims, VARLEN_PLAN_FWD, fwd_pairs(a.dims), a.dims.Hq, a.plan, a.status, st);
    if (e != cudaSuccess) return e;
  }
  p.o = a.o;
  p.o_res = a.o_res;
  p.lse = a.lse;
  p.status = a.status;
  p.counter = a.counter;
  p.timeout_ns = a.timeout_ns;
  p.total_units = fwd_units(a.dims);
  const bool split = MASK == MASK_NONE && !F8 && !VL && !SP && a.nsplit > 1;
  p.split0 = split ? a.split0 : p.total_units;
  p.nsplit = split ? a.nsplit : 1;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  if (split) p.total_units = a.split0 + (p.total_units - a.split0) * a.nsplit;
  const int grid = imax(1, imin(p.total_units, a.num_sms));
  p.trace = DG == DG_TRACE ? a.trace : nullptr;  // the host sets a.trace only when the grid fits TRACE_MAX_CTAS
  FwdSched sched;
  sched.on = 0;
  sched.grid = grid;
  if (a.sched != nullptr && a.sched->on && a.sched->grid == grid && !VL && !SP) sched = *a.sched;
  // launched with programmatic stream serialisation: the CTAs set up their barriers
  // and TMEM while the header-clearing kernel before them still runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, p, sched, a.tm_o, a.tm_r);
  if (e != cudaSuccess || !split) return e;
  // the combine, queued behind the forward with programmatic serialisation (its
  // CTAs wait in griddepcontrol.wait until the forward's parts are written)
  cfg.gridDim = dim3((fwd_units(a.dims) - a.split0) * 2 * TILE / (128 / (D / 8)));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, fwd_split_combine_kernel<D>, p);
}

// Zero a workspace header (status word, counters) and let the kernel after it
// start its set-up at once.
__global__ void __launch_bounds__(32) header_clear_kernel(uint4* h) {
  griddep_launch_dependents();
  if (threadIdx.x < FA_WS_HEADER_BYTES / 16) h[threadIdx.x] = make_uint4(0, 0, 0, 0);
}

}  // namespace

cudaError_t launch_header_clear(void* ws, cudaStream_t st) {
  header_clear_kernel<<<1, 32, 0, st>>>(static_cast<uint4*>(ws));
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t st) {
  const int m = mask_kind(a.dims);
  if (a.row_ptr != nullptr) {  // block-sparse: bf16, dense batch, no band
    if (a.sq != nullptr || a.dims.cu_q != nullptr || m == MASK_BAND) return cudaErrorInvalidValue;
    if (k_tiles(a.dims) > FwdLayout<128, false, true>::MAXL) return cudaErrorInvalidValue;
    if (a.d == 64)
      return m == MASK_CAUSAL ? launch_fwd_t<64, MASK_CAUSAL, false, false, true>(a, st)
                              : launch_fwd_t<64, MASK_NONE, false, false, true>(a, st);
    return m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL, false, false, true>(a, st)
                            : launch_fwd_t<128, MASK_NONE, false, false, true>(a, st);
  }
  if (a.dims.cu_q != nullptr) {  // packed sequences: bf16, no band
    if (a.sq != nullptr || m == MASK_BAND) return cudaErrorInvalidValue;
    if (a.d == 64)
      return m == MASK_CAUSAL ? launch_fwd_t<64, MASK_CAUSAL, false, true>(a, st)
                              : launch_fwd_t<64, MASK_NONE, false, true>(a, st);
    return m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL, false, true>(a, st)
                            : launch_fwd_t<128, MASK_NONE, false, true>(a, st);
  }
  if (a.sq != nullptr) {  // E4M3 operands (d = 128 only)
    if (a.d != 128) return cudaErrorInvalidValue;
    return m == MASK_BAND     ? launch_fwd_t<128, MASK_BAND, true>(a, st)
           : m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL, true>(a, st)
                              : launch_fwd_t<128, MASK_NONE, true>(a, st);
  }
  if (a.diag != DG_NONE) {  // timestamps, or the withheld hand-off: dense bf16 d = 128 only
    if (a.d != 128 || (a.diag == DG_TRACE && imin(fwd_units(a.dims), a.num_sms) > TRACE_MAX_CTAS))
      return cudaErrorInvalidValue;
    if (a.diag == DG_WITHHOLD)
      return m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL, false, false, false, DG_WITHHOLD>(a, st)
                              : launch_fwd_t<128, MASK_NONE, false, false, false, DG_WITHHOLD>(a, st);
    return m == MASK_BAND     ? launch_fwd_t<128, MASK_BAND, false, false, false, DG_TRACE>(a, st)
           : m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL, false, false, false, DG_TRACE>(a, st)
                              : launch_fwd_t<128, MASK_NONE, false, false, false, DG_TRACE>(a, st);
  }
  if (a.d == 64)
    return m == MASK_BAND ? launch_fwd_t<64, MASK_BAND>(a, st)
           : m == MASK_CAUSAL ? launch_fwd_t<64, MASK_CAUSAL>(a, st) : launch_fwd_t<64, MASK_NONE>(a, st);
  return m == MASK_BAND ? launch_fwd_t<128, MASK_BAND>(a, st)
         : m == MASK_CAUSAL ? launch_fwd_t<128, MASK_CAUSAL>(a, st) : launch_fwd_t<128, MASK_NONE>(a, st);
}

}  // namespace fa
