// Split-KV decode (FlashDecoding) and its log-sum-exp weighted combine.
//
// Method ("第18章 FlashAttention" §18.8.2; "CMU 11-868 L21" notes, slides
// 57-60): with a short query and a long KV cache, the cache is cut along its
// length into chunks that run in parallel; each chunk yields its own softmax
// statistics and partial output, and a second kernel merges them with weights
// e^{m_t - m}.  The query heads that share one K/V head, times the query
// positions, are packed into the rows of one matrix tile (GQA packing), so
// each K/V byte is read from HBM once for all of them.
//
// GB300 design.  The work is HBM-bound (4-16 flop per byte), so the kernel is
// built around the copy engine: one CTA per (split, K/V head, batch); a
// producer warp streams 128-key K and V tiles with TMA (16-byte aligned,
// 128-byte-swizzled boxes of 64 channels x 128 keys) through a ring of
// shared-memory stages; 8 compute warps share every tile.  The packed rows
// (Hq/Hkv * Nq of them) form RT = 1, 2 or 4 matrix tiles of 16 rows, which is
// what the warp-level mma.sync m16n8k16 handles: the warps split into RT
// groups, one per 16-row tile, and each warp of a group owns 16 RT keys of
// every 128-key tile; the scores, the online softmax and P stay in registers,
// and no cross-warp exchange is needed until the split ends.  (A 128-row
// tcgen05 product would be 50-87% padding here; lecture slides 57-60 pack the
// heads and the query positions into the rows in the same way.)  The warps'
// states are merged through shared memory into the split's (LSE_s, O_s); the
// combine kernel then merges the splits.
//
// Paged, variable-length cache (§18.8.2 part 3, §18.8.3: PagedAttention keeps
// the cache in fixed-size physical pages and maps each sequence's logical pages
// through a page table; each sequence has its own length).  The same kernel,
// with the producer resolving every 128-key tile through the page table: one
// TMA box per tile when a page holds whole tiles, else one box per page (pages
// of 16-64 keys stack into the tile with the same 128-byte swizzle, since each
// is a whole number of 8-row swizzle atoms).  Each sequence is split by its own
// length; splits past its end write an empty partial (LSE -inf, O 0).  Keys past
// the end of a sequence inside its last tile hold whatever the page (or an
// earlier tile) left in shared memory: their scores are masked and their V rows
// are zeroed in registers, so even NaN there cannot reach O.
//
// Head groups (HG).  A page holds all K/V heads of its rows side by side, so
// with small pages the per-head kernel needs eight 16-row boxes per 128-key
// tile and the copy engine's per-box cost, not HBM, sets the pace.  With HG =
// 8, 4 or 2 heads per CTA (Hkv a multiple of 8 and pages of whole 16-row
// slices; or Hkv a multiple of 4 or 2 and pages of 16-64 rows) one CTA serves
// HG K/V heads instead: a stage holds 128 / HG keys of all HG heads, loaded as
// boxes of rb = min(page, 128 / HG) rows x HG heads x 64 channels (lines
// head-major inside a box), so the stage has the size and the swizzle of a
// 128-key tile of one head.  Compute warp w works on head w % HG and on the
// 16-key slice w / HG of every stage, with its own softmax state; with HG = 8
// each warp's state is its head's partial, with HG = 4 or 2 the 2 or 4 warps of
// a head merge through shared memory as the per-head kernel's do.
#include <math.h>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float LN2 = 0.69314718055994530942f;
constexpr int WARPS = 8;              // compute warps
constexpr int MAX_ROW_TILES = 4;      // packed rows Hq/Hkv * Nq <= 64
static_assert(WARPS == DECODE_HEAD_GROUP, "the largest head group is one head per compute warp");
constexpr int THREADS = 32 * (WARPS + 1);

template <int D>
struct DecLayout {
  static constexpr int TB = TILE * D * 2;   // one K or V tile
  static constexpr int STAGES = D == 64 ? 6 : 3;
  static constexpr int OFF_KV = 0;          // stage s: K at s*2*TB, V at s*2*TB + TB
  static constexpr int OFF_BAR = STAGES * 2 * TB;
  static constexpr int BYTES = OFF_BAR + 2 * STAGES * 8 + 64;
  static constexpr int ALLOC = BYTES + 1024;
  // after the pipeline ends the stage memory holds the per-warp states:
  // m[WARPS][16], l[WARPS][16], o[WARPS][16][D]  (fp32)
  static_assert(WARPS * 16 * (2 + D) * 4 <= STAGES * 2 * TB, "merge area");
};

struct DecParams {
  Dims dims;
  int d;
  float scale_log2;
  const __nv_bfloat16* q;
  int64_t q_sb, q_sn, q_sh;
  float* lse_part;
  float* o_part;
  int num_splits, chunk;
  int* status;
  unsigned long long timeout_ns;
  const int* block_table;  // paged: [B, max_pages]
  int max_pages;
  const int* seqlens;      // paged: [B]
  int num_pages, page_size;
};

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Byte offset of (key, channel) inside a TMA tile of 128 keys x D channels
// stored as D/64 boxes of [128 keys][128 bytes] with the 128-byte swizzle
// (16-byte chunk index XOR key % 8).
__device__ __forceinline__ uint32_t swz(int key, int ch) {
  return (ch >> 6) * (TILE * 128) + key * 128 + ((((ch & 63) >> 3) ^ (key & 7)) << 4) + ((ch & 7) << 1);
}

template <int D, bool PAGED, int HGK, int RT>
__global__ void __launch_bounds__(THREADS, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecParams p) {
  using L = DecLayout<D>;
  constexpr bool HG = HGK > 0;  // HGK K/V heads per CTA, or one head (0)
  static_assert(!HG || PAGED, "head groups are a paged layout");
  static_assert(!HG || RT == 1, "a head group has one 16-row tile per head");
  static_assert(HGK == 0 || HGK == 2 || HGK == 4 || HGK == WARPS, "heads per CTA");
  constexpr int WPR = WARPS / RT;  // warps per 16-row tile
  constexpr int KW = TILE / WPR;   // keys of each 128-key tile per warp (16 RT), in RT chunks of 16
  constexpr int SPS = HG ? WARPS / HGK : 1;  // (HG) 16-key slices per stage = warps per head
  constexpr int KT = HG ? 16 * SPS : TILE;   // keys per stage (of each head of the CTA)
  constexpr bool MERGE = !HG || SPS > 1;     // several warps hold parts of one row
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + L::STAGES;
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int split = blockIdx.x, b = blockIdx.z;
  const int hw = HG && warp < WARPS ? warp % HGK : 0;  // (HG) this warp's head in the group
  const int js = HG && warp < WARPS ? warp / HGK : 0;  // (HG) this warp's 16-key slice of each stage
  const int kvh = HG ? blockIdx.y * HGK + hw : blockIdx.y;  // this warp's K/V head
  const Dims& s = p.dims;
  const int g = s.Hq / s.Hkv;
  const int rows = g * s.Nq;
  const Ctl ctl{p.status, p.timeout_ns};
  int len = s.Nk, chunk = p.chunk;  // this sequence's keys and its split length
  if (PAGED) {
    len = p.seqlens[b];
    if (len < 1 || len > s.Nk) {
      if (threadIdx.x == 0 && split == 0 && kvh == 0) report(ctl, FA_STATUS_BAD_INPUT);
      len = imax(0, imin(len, s.Nk));
    }
    chunk = cdiv(cdiv(len, KT), p.num_splits) * KT;
  }
  const int rb = HG ? imin(p.page_size, KT) : 0;  // (HG) rows of a box: KT, or a whole page
  const int k0 = split * chunk;
  const int k1 = imin(len, k0 + chunk);
  const int ntiles = k1 > k0 ? cdiv(k1 - k0, KT) : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], WARPS);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();

  if (warp == WARPS) {  // ---------------------------------------------- producer
    if (HG) {
      // Stage t: keys [k0 + t KT, + KT) of heads HGK blockIdx.y .. + HGK-1, as boxes of rb
      // rows (a page's rows r .. r + rb - 1; rb divides the page) x HGK heads x 64
      // channels; lane i reads the page of box i one stage ahead and loads it.  No box
      // is loaded past the split's end, where the table need not be valid.
      // Coordinates of the map: (channel, row, head, page).
      const int64_t trow = static_cast<int64_t>(b) * p.max_pages;
      auto page_of = [&](int t) {
        const int key = k0 + t * KT + lane * rb;
        if (t >= ntiles || lane * rb >= KT || key >= k1) return -1;
        int pg = p.block_table[trow + key / p.page_size];
        if (pg < 0 || pg >= p.num_pages) {  // reads as zeros (out-of-range TMA box); reported
          report(ctl, FA_STATUS_BAD_INPUT);
          pg = p.num_pages;
        }
        return pg;
      };
      int issued = 0;
      int next_page = page_of(0);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % L::STAGES;
        const int page = next_page;
        next_page = page_of(t + 1);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((t / L::STAGES) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int kk = k0 + t * KT;
        const int nbox = imin(KT / rb, cdiv(k1 - kk, rb));
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 4 * nbox * rb * HGK * D);  // K and V boxes
        __syncwarp();
        if (lane < nbox) {
          uint8_t* dst = smem + L::OFF_KV + st * 2 * L::TB + lane * rb * HGK * 128;
          const int row = (kk + lane * rb) % p.page_size;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(dst + c * (TILE * 128), &tm_k, &full[st], c * 64, row, blockIdx.y * HGK, page);
            tma_load_4d(dst + L::TB + c * (TILE * 128), &tm_v, &full[st], c * 64, row, blockIdx.y * HGK, page);
          }
        }
        ++issued;
      }
      if (lane == 0)
        for (int t = imax(0, issued - L::STAGES); t < issued; ++t)
          mbar_wait(&full[t % L::STAGES], (t / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
      if (!MERGE) return;  // one warp per head: the compute warps do not merge, no block barrier follows
    } else if (!PAGED) {
      if (lane == 0) {
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
          const int st = t % L::STAGES;
          if (!mbar_wait(&empty[st], ((t / L::STAGES) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) break;
          uint8_t* dst = smem + L::OFF_KV + st * 2 * L::TB;
          const int kk = k0 + t * TILE;  // first key of the tile
          mbar_arrive_expect_tx(&full[st], 2 * L::TB);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(dst + c * (TILE * 128), &tm_k, &full[st], c * 64, kvh, kk, b);
            tma_load_4d(dst + L::TB + c * (TILE * 128), &tm_v, &full[st], c * 64, kvh, kk, b);
          }
          ++issued;
        }
        // wait for the copies in flight before the CTA may exit
        for (int t = imax(0, issued - L::STAGES); t < issued; ++t)
          mbar_wait(&full[t % L::STAGES], (t / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
      }
    } else {
      // The whole warp: lane i reads the page of box i of a tile and loads that box,
      // so a tile's page-table reads go out together, one tile ahead of its loads.
      // Boxes hold `rows_box` keys: one page (or a whole tile when pages hold whole
      // tiles); none is loaded past the sequence's end, where the table need not be valid.
      const int rows_box = imin(p.page_size, TILE);
      const int64_t trow = static_cast<int64_t>(b) * p.max_pages;
      auto page_of = [&](int t) {
        const int off = lane * rows_box, key = k0 + t * TILE + off;
        if (t >= ntiles || off >= TILE || key >= len) return -1;
        int pg = p.block_table[trow + key / p.page_size];
        if (pg < 0 || pg >= p.num_pages) {  // reads as zeros (out-of-range TMA box); reported
          report(ctl, FA_STATUS_BAD_INPUT);
          pg = p.num_pages;
        }
        return pg;
      };
      int issued = 0;
      int next_page = page_of(0);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % L::STAGES;
        const int page = next_page;
        next_page = page_of(t + 1);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((t / L::STAGES) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int kk = k0 + t * TILE;
        const int nbox = imin(TILE / rows_box, cdiv(len - kk, rows_box));
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 4 * nbox * rows_box * D);  // K and V boxes
        __syncwarp();
        if (lane < nbox) {
          uint8_t* dst = smem + L::OFF_KV + st * 2 * L::TB + lane * rows_box * 128;
          const int row = (kk + lane * rows_box) % p.page_size;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(dst + c * (TILE * 128), &tm_k, &full[st], c * 64, kvh, row, page);
            tma_load_4d(dst + L::TB + c * (TILE * 128), &tm_v, &full[st], c * 64, kvh, row, page);
          }
        }
        ++issued;
      }
      if (lane == 0)
        for (int t = imax(0, issued - L::STAGES); t < issued; ++t)
          mbar_wait(&full[t % L::STAGES], (t / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
    }
    __syncwarp();     // lanes 1-31 wait for lane 0's drain: the barrier needs the whole warp
    __syncthreads();  // pairs with the compute warps' barrier before the merge
    __syncthreads();
    return;
  }

  // -------------------------------------------------------------- compute warps
  const int gq = lane >> 2, tq = lane & 3;  // fragment row group / column pair
  const int rt = warp / WPR;                // this warp's 16-row tile (HG: 0)
  // Q as m16n8k16 A fragments (rows r = qpos * g + head-in-group, zero above `rows`).
  uint32_t qa[D / 16][4];
  {
    const int row_a = rt * 16 + gq, row_b = row_a + 8;  // this thread's two fragment rows
    const __nv_bfloat16* qpa = nullptr;
    const __nv_bfloat16* qpb = nullptr;
    if (row_a < rows) qpa = p.q + b * p.q_sb + (row_a / g) * p.q_sn + (kvh * g + row_a % g) * p.q_sh;
    if (row_b < rows) qpb = p.q + b * p.q_sb + (row_b / g) * p.q_sn + (kvh * g + row_b % g) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = ks * 16 + 2 * tq;
      qa[ks][0] = qpa ? *reinterpret_cast<const uint32_t*>(qpa + c0) : 0u;
      qa[ks][1] = qpb ? *reinterpret_cast<const uint32_t*>(qpb + c0) : 0u;
      qa[ks][2] = qpa ? *reinterpret_cast<const uint32_t*>(qpa + c0 + 8) : 0u;
      qa[ks][3] = qpb ? *reinterpret_cast<const uint32_t*>(qpb + c0 + 8) : 0u;
    }
  }
  const float c = p.scale_log2;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  const int mat = lane >> 3, mrow = lane & 7;  // ldmatrix: which 8x8 matrix this lane addresses
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % L::STAGES;
    ok = mbar_wait(&full[st], (t / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint32_t kb = smem_u32(smem + L::OFF_KV + st * 2 * L::TB);
    const uint32_t vb = kb + L::TB;
    // this warp's lines of the stage: keys KW (warp % WPR) .. + KW-1 of the tile, or
    // (HG) the 16 keys of slice js of head hw, inside box (16 js) / rb
    const int key_base = HG ? (16 * js / rb) * rb * HGK + hw * rb + (16 * js) % rb : KW * (warp % WPR);

    // S = Q K^T for 16 rows x KW keys (2 RT n8 tiles)
    float sacc[2 * RT][4];
#pragma unroll
    for (int nt = 0; nt < 2 * RT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int cq = 0; cq < RT; ++cq)
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        // matrices: (keys 0-7, ch lo), (keys 0-7, ch hi), (keys 8-15, ch lo), (keys 8-15, ch hi)
        const int key = key_base + 16 * cq + 8 * (mat >> 1) + mrow;
        const int ch = ks * 16 + 8 * (mat & 1);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kb + swz(key, ch), b00, b01, b10, b11);
        mma_16816(sacc[2 * cq], qa[ks], b00, b01);
        mma_16816(sacc[2 * cq + 1], qa[ks], b10, b11);
      }
    // mask keys outside [k0, k1)
    const int key0 = k0 + t * KT + (HG ? 16 * js : key_base);
    float sv[2 * RT][4];
#pragma unroll
    for (int nt = 0; nt < 2 * RT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = key0 + 8 * nt + 2 * tq + (i & 1);
        sv[nt][i] = key < k1 ? sacc[nt][i] : -INFINITY;
      }
    // online softmax for rows gq (i = 0,1) and gq+8 (i = 2,3), over the warp's KW keys
    uint32_t pa[RT][4];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2 * RT; ++nt) mx = fmax3(mx, sv[nt][2 * hr], sv[nt][2 * hr + 1]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_tile = mx * c;
      const float m_new = fmaxf(m_run[hr], m_tile);
      const float alpha = (m_new == m_run[hr]) ? 1.f : ex2(m_run[hr] - m_new);
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      float lsum = 0.f;
#pragma unroll
      for (int cq = 0; cq < RT; ++cq) {
        const float p00 = ex2(fmaf(sv[2 * cq][2 * hr], c, -mu)), p01 = ex2(fmaf(sv[2 * cq][2 * hr + 1], c, -mu));
        const float p10 = ex2(fmaf(sv[2 * cq + 1][2 * hr], c, -mu));
        const float p11 = ex2(fmaf(sv[2 * cq + 1][2 * hr + 1], c, -mu));
        lsum += (p00 + p01 + p10 + p11);
        pa[cq][hr] = pack_bf16(p00, p01);      // a0 (row gq) / a1 (row gq+8): keys 2tq, 2tq+1 of the chunk
        pa[cq][2 + hr] = pack_bf16(p10, p11);  // a2 / a3: keys 8+2tq, 9+2tq
      }
      l_run[hr] = l_run[hr] * alpha + lsum;
      m_run[hr] = m_new;
      if (alpha != 1.f) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o[nt][2 * hr] *= alpha;
          o[nt][2 * hr + 1] *= alpha;
        }
      }
    }
    // O += P V: B fragments of V (16 keys x 8 channels) via transposed ldmatrix,
    // one 16-key chunk at a time.  Paged: V rows past the split's end may hold
    // anything (stale shared memory or an unused part of a page); they are zeroed,
    // as their P is.  This thread's fragment halves cover keys kc + 2tq (+1) and
    // kc + 8 + 2tq (+1) of chunk kc.
#pragma unroll
    for (int cq = 0; cq < RT; ++cq) {
      uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
      const int kc = key0 + 16 * cq;
      if (PAGED && kc + 16 > k1) {
        const int ka = kc + 2 * tq, kb8 = ka + 8;
        vmask_lo = (ka < k1 ? 0x0000ffffu : 0u) | (ka + 1 < k1 ? 0xffff0000u : 0u);
        vmask_hi = (kb8 < k1 ? 0x0000ffffu : 0u) | (kb8 + 1 < k1 ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        // matrices: (keys 0-7, ch n0..), (keys 8-15, ch n0..), (keys 0-7, ch n0+8..), (keys 8-15, ch n0+8..)
        const int key = key_base + 16 * cq + 8 * (mat & 1) + mrow;
        const int ch = np * 16 + 8 * (mat >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vb + swz(key, ch), v0, v1, v2, v3);
        if (PAGED) {
          v0 &= vmask_lo;
          v2 &= vmask_lo;
          v1 &= vmask_hi;
          v3 &= vmask_hi;
        }
        mma_16816(o[2 * np], pa[cq], v0, v1);
        mma_16816(o[2 * np + 1], pa[cq], v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---------------------------------------------------------- merge the 8 warps
  // row sums are spread over the 4 lanes of a quad
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
  if (!MERGE) {  // one warp per head: its state is the split's (rows gq and gq + 8)
    if (!ok) return;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = gq + 8 * hr;
      if (row >= rows) continue;
      const float l = l_run[hr];
      const float inv = l > 0.f ? 1.f / l : 0.f;  // an empty split: O 0, LSE -inf
      const int qpos = row / g, hq = kvh * g + row % g;
      const int64_t prow = ((static_cast<int64_t>(b) * s.Hq + hq) * s.Nq + qpos) * p.num_splits + split;
      float* op = p.o_part + prow * D + 2 * tq;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt)
        *reinterpret_cast<float2*>(op + nt * 8) = make_float2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
      if (tq == 0) p.lse_part[prow] = l > 0.f ? (m_run[hr] + __log2f(l)) * LN2 : -INFINITY;
    }
    return;
  }
  // all compute warps and the producer must be past the pipeline before the
  // stage memory is reused
  __syncthreads();
  float* sm = reinterpret_cast<float*>(smem);
  float* sm_m = sm;                       // [WARPS][16]
  float* sm_l = sm + WARPS * 16;          // [WARPS][16]
  float* sm_o = sm + 2 * WARPS * 16;      // [WARPS][16][D]
  if (tq == 0) {
    sm_m[warp * 16 + gq] = m_run[0];
    sm_m[warp * 16 + gq + 8] = m_run[1];
    sm_l[warp * 16 + gq] = l_run[0];
    sm_l[warp * 16 + gq + 8] = l_run[1];
  }
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int ch = nt * 8 + 2 * tq;
    sm_o[(warp * 16 + gq) * D + ch] = o[nt][0];
    sm_o[(warp * 16 + gq) * D + ch + 1] = o[nt][1];
    sm_o[(warp * 16 + gq + 8) * D + ch] = o[nt][2];
    sm_o[(warp * 16 + gq + 8) * D + ch + 1] = o[nt][3];
  }
  __syncthreads();
  if (!ok) return;
  // 256 threads: thread -> (16-row group, local row, channel range).  A group is a
  // 16-row tile of the packed rows (its state in the WPR warps of that tile) or
  // (HG) one head (its state in warps head, head + HGK, ...), at local row lr.
  constexpr int NW = HG ? SPS : WPR;         // warps holding parts of one row
  constexpr int GROUPS = HG ? HGK : RT;
  constexpr int PER = GROUPS * 16 * D / 256;  // channels per thread
  const int tid = threadIdx.x;               // < 256
  const int grow = tid / (D / PER);
  const int grp = grow / 16, lr = grow % 16;
  const int row = HG ? lr : grow;            // the packed row of the group's head
  const int chb = (tid % (D / PER)) * PER;
  auto wid = [&](int w) { return HG ? grp + HGK * w : grp * WPR + w; };
  if (row < rows) {
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mstar = fmaxf(mstar, sm_m[wid(w) * 16 + lr]);
    const float mref = mstar == -INFINITY ? 0.f : mstar;
    float wsum = 0.f, wt[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = sm_m[wid(w) * 16 + lr];
      wt[w] = mw == -INFINITY ? 0.f : ex2(mw - mref);
      wsum += wt[w] * sm_l[wid(w) * 16 + lr];
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;  // an empty split: O 0, LSE -inf
    const int head = HG ? blockIdx.y * HGK + grp : kvh;
    const int qpos = row / g, hq = head * g + row % g;
    const int64_t prow = ((static_cast<int64_t>(b) * s.Hq + hq) * s.Nq + qpos) * p.num_splits + split;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) acc += wt[w] * sm_o[(wid(w) * 16 + lr) * D + chb + i];
      p.o_part[prow * D + chb + i] = acc * inv;
    }
    if (chb == 0) p.lse_part[prow] = wsum > 0.f ? (mref + __log2f(wsum)) * LN2 : -INFINITY;
  }
}

// One warp per output row: LSE = ln sum_s e^{LSE_s}; O = sum_s e^{LSE_s - LSE} O_s.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const float* __restrict__ lse_part,
                                                                const float* __restrict__ o_part, OutRows o,
                                                                float* __restrict__ lse, int rows_total, int Hq,
                                                                int Nq, int S) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows_total) return;
  const float* lp = lse_part + static_cast<int64_t>(row) * S;
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float mxs = mx == -INFINITY ? 0.f : mx;  // no split saw a key: O 0, LSE -inf
  float den = 0.f;
  for (int s = lane; s < S; s += 32) den += __expf(lp[s] - mxs);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float lse_row = mxs + __logf(den);
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  const float* op = o_part + static_cast<int64_t>(row) * S * D;
  for (int s = 0; s < S; ++s) {
    const float w = den > 0.f ? __expf(lp[s] - lse_row) : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] += w * op[s * D + lane * PER + i];
  }
  // row = (b * Hq + h) * Nq + qpos
  const int qpos = row % Nq, bh = row / Nq, h = bh % Hq, b = bh / Hq;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(o.ptr) + b * o.sb + static_cast<int64_t>(qpos) * o.sn +
                       h * o.sh + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16(acc[i], acc[i + 1]);
  if (lane == 0) lse[row] = lse_row;
}

template <int D, int RT>
cudaError_t launch_decode_t(const DecodeLaunch& a, cudaStream_t st) {
  using L = DecLayout<D>;
  auto kern = a.block_table == nullptr ? fa_decode_split_kernel<D, false, 0, RT>
               : a.head_group == 8   ? fa_decode_split_kernel<D, true, 8, 1>
               : a.head_group == 4   ? fa_decode_split_kernel<D, true, 4, 1>
               : a.head_group == 2   ? fa_decode_split_kernel<D, true, 2, 1>
                                     : fa_decode_split_kernel<D, true, 0, RT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  DecParams p;
  p.dims = a.dims;
  p.d = a.d;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.q_sb = a.q_sb;
  p.q_sn = a.q_sn;
  p.q_sh = a.q_sh;
  p.lse_part = a.lse_part;
  p.o_part = a.o_part;
  p.num_splits = a.num_splits;
  p.chunk = a.chunk;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.block_table = a.block_table;
  p.max_pages = a.max_pages;
  p.seqlens = a.seqlens;
  p.num_pages = a.num_pages;
  p.page_size = a.page_size;
  dim3 grid(a.num_splits, a.head_group ? a.dims.Hkv / a.head_group : a.dims.Hkv, a.dims.B);
  kern<<<grid, THREADS, L::ALLOC, st>>>(a.tm_k, a.tm_v, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows_total = a.dims.B * a.dims.Hq * a.dims.Nq;
  fa_decode_combine_kernel<D><<<cdiv(rows_total, 4), 128, 0, st>>>(a.lse_part, a.o_part, a.o, a.lse, rows_total,
                                                                   a.dims.Hq, a.dims.Nq, a.num_splits);
  return cudaGetLastError();
}

}  // namespace

// Packed rows Hq/Hkv * Nq in 16-row tiles: 1, 2 or 4 (head groups: 1).
int decode_row_tiles(const Dims& d) { return cdiv((d.Hq / d.Hkv) * d.Nq, 16); }

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t st) {
  const int rt = decode_row_tiles(a.dims);
  if (rt > MAX_ROW_TILES) return cudaErrorInvalidValue;
  if (a.head_group && (rt != 1 || a.block_table == nullptr || a.dims.Hkv % a.head_group != 0 ||
                       (a.head_group != 2 && a.head_group != 4 && a.head_group != WARPS)))
    return cudaErrorInvalidValue;
  if (a.d == 64)
    return rt == 1 ? launch_decode_t<64, 1>(a, st) : rt == 2 ? launch_decode_t<64, 2>(a, st) : launch_decode_t<64, 4>(a, st);
  return rt == 1 ? launch_decode_t<128, 1>(a, st) : rt == 2 ? launch_decode_t<128, 2>(a, st) : launch_decode_t<128, 4>(a, st);
}

}  // namespace fa
