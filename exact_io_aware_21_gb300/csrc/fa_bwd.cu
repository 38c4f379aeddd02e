// Backward kernels: attention gradients with P rebuilt on chip.
//
// Method ("第18章 FlashAttention" §18.4.4, Fig. 18-17; "CMU 11-868 L21" notes,
// slide 14): the forward pass saved only O and the row statistic (here the
// log-sum-exp); the backward pass recomputes S = Q K^T tile by tile, rebuilds
// P = exp(scale S - LSE) with no rescaling, and forms dV = P^T dO,
// dP = dO V^T, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
// D_i = rowsum(P o dP) over the whole row equals dO_i . O_i, so it is computed
// once, before the tile loops, by the preprocess kernel.
//
// GB300 design: three kernels and no atomics, so results are deterministic.
//   preprocess  D = rowsum(dO o O) and LSE * log2(e), both padded to whole
//               128-row tiles (+inf / 0 in the padding, which zeroes P there).
//   dK/dV       one CTA per SM, persistent; a unit is one 128-key tile of one
//               K/V head; it loops over the query heads of the group and their
//               query tiles (causal: only tiles at or below the diagonal).
//               TMEM: S^T [0,128) dP^T [128,256) dV [256,256+d) dK [256+d,..);
//               at d = 64 a second S^T buffer [384,512) takes every other
//               iteration.  P^T and dS^T are written back over S^T and dP^T as
//               bf16 and feed the dV and dK products from TMEM.
//   dQ          a unit is one 128-row query tile; it loops over key tiles.
//   Dense path: the three follow a header-clearing kernel, each launched with
//   programmatic stream serialisation: it sets up while the one before it
//   finishes and waits (griddepcontrol) before reading that one's results.  The
//   dK/dV kernel lets the dQ kernel launch as soon as its own wait is over, so
//   dQ CTAs take over SMs as dK/dV CTAs finish; dQ reads only the preprocess
//   kernel's output, complete by then, and skips its wait in that case.
//               TMEM: S double-buffered [0,256), dP [256,384), dQ [384,384+d);
//               dS is written over dP as bf16 and feeds dQ += dS K.
// Warp roles: warp 0 loads with TMA, one thread of warp 1 issues tcgen05 MMAs,
// and two warpgroups (warps 4-7 and 8-11) do the elementwise work: both hold
// the same 128 rows (one TMEM lane per thread) and split the 128 columns,
// warpgroup 0 taking columns 0-63 and warpgroup 1 columns 64-127.  Each writes
// its bf16 half (P^T or dS) back into TMEM columns it has itself already read:
// the half for columns 0-63 at column offset 0, the half for 64-127 at offset
// 64, so the two warpgroups never wait for each other; the MMAs that read that
// operand from TMEM address its second half 64 columns on.
#include <math.h>

#include <utility>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

struct BwdParams {
  Dims dims;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  OutRows o, o_res, dout, dq, dk, dv;
  const float* lse;
  float* neg_lse2;   // -LSE * log2(e) per query row (-inf in padding)
  float* neg_delta;  // -D per query row
  int nq_pad;
  int* status;
  int* counter;
  unsigned long long timeout_ns;
  int total_units;
  const int* plan;  // packed sequences: the kernel's device-side work plan (units with work only)
  const int* rows_ptr;  // block-sparse: key tiles of each query tile (ascending) ...
  const int* rows_idx;
  const int* cols_ptr;  // ... and query tiles of each key tile (ascending)
  const int* cols_idx;
  const int* sp_plan;   // block-sparse: the dK/dV segment plan
  float* sp_pool;       // ... and the partial tiles of split key tiles
  int tma_out;          // dense: dK and dV leave through TMA stores
  int dq_after_dkdv;    // dQ launched right after the dK/dV kernel of the same call (see launch_bwd_t)
};

// ================================================================== preprocess
// threads per row = D / 8 (one 16-byte chunk of dO and of O each)
// One row's D and -LSE2 (TPR threads; `part` = this thread's 16-byte chunk).
// Rows at or past the sequence's length get D = 0 and -LSE2 = -inf (P = 0).
template <int D, bool VL>
__device__ __forceinline__ void preprocess_row(const BwdParams& p, int b, int h, int q, int64_t row, int part) {
  constexpr int TPR = D / 8;
  const SeqRows sr = seq_rows<VL>(p.dims, b);
  const int nq = sr.s.Nq;                       // this sequence's rows
  const int64_t qrow = sr.qoff + static_cast<int64_t>(q);
  float acc = 0.f;
  if (q < nq) {
    // all three loads go out before any use (one memory round trip per row)
    const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(p.o.ptr) + b * p.o.sb + qrow * p.o.sn +
                             h * p.o.sh + part * 8;
    const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(p.dout.ptr) + b * p.dout.sb +
                             qrow * p.dout.sn + h * p.dout.sh + part * 8;
    const bool res = p.o_res.ptr != nullptr;  // D = dO . (O + residual)
    const __nv_bfloat16* rr = res ? reinterpret_cast<const __nv_bfloat16*>(p.o_res.ptr) + b * p.o_res.sb +
                                        qrow * p.o_res.sn + h * p.o_res.sh + part * 8
                                  : o;
    // O and the residual are not read again (streaming loads); dO is, by the
    // dK/dV and dQ kernels that follow, so it is loaded the ordinary way
    const uint4 ov = __ldcs(reinterpret_cast<const uint4*>(o));
    const uint4 gv = *reinterpret_cast<const uint4*>(g);
    const uint4 rv = res ? __ldcs(reinterpret_cast<const uint4*>(rr)) : make_uint4(0, 0, 0, 0);
    const uint32_t* ou = reinterpret_cast<const uint32_t*>(&ov);
    const uint32_t* gu = reinterpret_cast<const uint32_t*>(&gv);
    const uint32_t* ru = reinterpret_cast<const uint32_t*>(&rv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = unpack_bf16(ou[i]), c = unpack_bf16(gu[i]);
      acc = fmaf(a.x, c.x, acc);
      acc = fmaf(a.y, c.y, acc);
    }
    if (res) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 e = unpack_bf16(ru[i]), c = unpack_bf16(gu[i]);
        acc = fmaf(e.x, c.x, acc);
        acc = fmaf(e.y, c.y, acc);
      }
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
  if (part == 0) {
    p.neg_delta[row] = -acc;
    // LSE [B, Hq, Nq], or [Hq, total_q] for packed sequences
    const int64_t li = VL ? static_cast<int64_t>(h) * p.dims.total_q + qrow
                          : (static_cast<int64_t>(b) * p.dims.Hq + h) * p.dims.Nq + q;
    p.neg_lse2[row] = q < nq ? -p.lse[li] * LOG2E : -INFINITY;
  }
}

// Dense: one thread group per row of the padded [B * Hq, nq_pad] layout.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  griddep_wait();  // launched with programmatic serialisation after the header clear
  griddep_launch_dependents();
  constexpr int TPR = D / 8;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) / TPR;
  const int64_t rows = static_cast<int64_t>(p.dims.B) * p.dims.Hq * p.nq_pad;
  if (row >= rows) return;
  const int q = static_cast<int>(row % p.nq_pad);
  const int bh = static_cast<int>(row / p.nq_pad);
  preprocess_row<D, false>(p, bh / p.dims.Hq, bh % p.dims.Hq, q, row, threadIdx.x % TPR);
}

// Packed sequences: only the query tiles that exist (the dQ plan's units); rows
// of the max-length padding that no kernel reads are left alone.  One block per
// RPP rows of a unit, over a host-side bound on the unit count: blocks past the
// plan's count return at once.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_varlen_kernel(const BwdParams p, const int* plan_dq) {
  constexpr int TPR = D / 8, RPP = 256 / TPR;  // threads per row, rows per block
  constexpr int BPU = TILE / RPP;              // blocks per unit
  const int u = blockIdx.x / BPU;
  if (u >= __ldg(plan_dq)) return;
  int b, h, qt;
  plan_unit(plan_dq, p.dims.Hq, u, b, h, qt);
  const int r = (blockIdx.x % BPU) * RPP + threadIdx.x / TPR;
  const int64_t row0 = (static_cast<int64_t>(b) * p.dims.Hq + h) * p.nq_pad + qt * TILE;
  preprocess_row<D, true>(p, b, h, qt * TILE + r, row0 + r, threadIdx.x % TPR);
}

// ================================================================== shared helpers
// EW: called by a whole converged warp, one elected lane issuing each MMA (else
// by a single lane).
template <int D, bool EW = false>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t IDESC = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = (k / 4) * (TILE * 128) + (k % 4) * 32;
    const uint64_t ad = sdesc_sw128(a_base + off, 16, 1024), bd = sdesc_sw128(b_base + off, 16, 1024);
    if (!EW || elect_one()) mma_ss(d_tmem, ad, bd, IDESC, k > 0);
  }
}

// D[128 x D] (+)= A[tmem, 128 x 128 bf16] * B[smem tile 128 x D, N-major].
// A's K columns 0-63 are packed at TMEM columns [0, 32), K columns 64-127 at
// [64, 96) (one half per elementwise warpgroup).
template <int D, bool EW = false>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, bool acc) {
  constexpr uint32_t IDESC = idesc_bf16(128, D, false, true);
#pragma unroll
  for (int k = 0; k < TILE / 16; ++k) {
    const uint64_t bd = sdesc_sw128(b_base + k * 16 * 128, TILE * 128, 1024);
    if (!EW || elect_one()) mma_ts(d_tmem, a_tmem + k * 8 + (k >= 4 ? 32 : 0), bd, IDESC, (acc || k > 0) ? 1u : 0u);
  }
}

// Half of issue_ts: the four K steps whose A columns come from chunk `half` of
// each elementwise warpgroup (K steps 0,1,4,5 for half 0; 2,3,6,7 for half 1),
// so the product can start on the columns written first.
template <int D, int HALF, bool EW = false>
__device__ __forceinline__ void issue_ts_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, bool acc) {
  constexpr uint32_t IDESC = idesc_bf16(128, D, false, true);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int k = (i & 1) + 2 * HALF + (i >> 1) * 4;
    const uint64_t bd = sdesc_sw128(b_base + k * 16 * 128, TILE * 128, 1024);
    if (!EW || elect_one()) mma_ts(d_tmem, a_tmem + k * 8 + (k >= 4 ? 32 : 0), bd, IDESC, (acc || i > 0) ? 1u : 0u);
  }
}

// Store accumulator columns [col0, col0 + NC) of the warp's 32 TMEM lanes as bf16
// rows (times mul): dst0 = element (lane 0's row, column 0); rows at or beyond
// `live` (counted from lane 0) are skipped.  scratch == nullptr: direct stores.
template <int NC>
__device__ __forceinline__ void store_acc_rows(uint32_t t_acc, int col0, float mul, __nv_bfloat16* dst0,
                                               int64_t stride, int live, uint8_t* scratch) {
  const float2 m2 = make_float2(mul, mul);
#pragma unroll
  for (int cc = 0; cc < NC / 32; ++cc) {
    uint32_t v[32];
    tmem_ld32(t_acc + col0 + cc * 32, v);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = __fmul2_rn(f32x2(v[2 * i], v[2 * i + 1]), m2);
      w[i] = pack_bf16(f.x, f.y);
    }
    if (scratch != nullptr) {
      store_rows32_bf16(w, scratch, dst0 + col0 + cc * 32, stride, live);
    } else if (lane_id() < live) {  // no scratch: each lane stores its own row
      uint4* d4 = reinterpret_cast<uint4*>(dst0 + lane_id() * stride + col0 + cc * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

// Store accumulator columns [col0, col0 + NC) of this thread's TMEM lane as fp32 at dst.
template <int NC>
__device__ __forceinline__ void store_acc_f32(uint32_t t_acc, int col0, float* dst) {
#pragma unroll
  for (int cc = 0; cc < NC / 32; ++cc) {
    uint32_t v[32];
    tmem_ld32(t_acc + col0 + cc * 32, v);
    uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) d4[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// Accumulator columns [col0, col0 + NC) of the warp's 32 TMEM lanes as bf16 (times
// mul), leaving through TMA stores of 32 x 32 boxes at (col0 + 32 c, c1, c2, c3) of
// `map`: each box is staged in `buf` (2 KB, 512-byte aligned) in the 64-byte-swizzled
// layout (16-byte chunk q of row r at chunk q ^ ((r / 2) % 4)); the store made from the
// buffer before must have read it first.  Rows past the tensor's end are dropped by
// the copy engine.
template <int NC>
__device__ __forceinline__ void store_acc_boxes(uint32_t t_acc, int col0, float mul, const CUtensorMap* map,
                                                int c1, int c2, int c3, uint8_t* buf) {
  const float2 m2 = make_float2(mul, mul);
  const int lr = lane_id();
#pragma unroll 1
  for (int cc = 0; cc < NC / 32; ++cc) {
    uint32_t v[32];
    tmem_ld32(t_acc + col0 + cc * 32, v);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = __fmul2_rn(f32x2(v[2 * i], v[2 * i + 1]), m2);
      w[i] = pack_bf16(f.x, f.y);
    }
    if (lr == 0) bulk_wait_read<0>();
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(buf + lr * 64 + ((q ^ ((lr >> 1) & 3)) << 4)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lr == 0) {
      tma_store_4d(map, buf, col0 + cc * 32, c1, c2, c3);
      bulk_commit();
    }
  }
}

// ================================================================== dK / dV
template <int D>
struct DkvLayout {
  static constexpr int TB = TILE * D * 2;
  static constexpr int STAGES = D == 64 ? 4 : 2;
  static constexpr int STAGE = 2 * TB + 1024;  // Q_i, dO_i, -lse2[128], -D[128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TB;
  static constexpr int OFF_ST = 2 * TB;
  // S^T buffers: at d = 64, TMEM's last 128 columns hold a second one, so the
  // S^T of an iteration two ahead is computed while this one's P^T is still in use
  static constexpr int SB = D == 64 ? 2 : 1;
  static constexpr int OFF_BAR = OFF_ST + STAGES * STAGE;
  // unit_full[2] unit_empty[2] kv_full kv_empty st_full[S] st_empty[S] s_full[2] dp_full p_full[2] ds_full
  // acc_full
  static constexpr int NBAR = 4 + 2 + 2 * STAGES + 7;
  static constexpr int OFF_UNIT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_TMEM = OFF_UNIT + 16;
  // row-store scratch, one per gradient warp; 1024-byte aligned, so that each warp's
  // first 2 KB (at a multiple of 2560 bytes) can stage a swizzled TMA-store box
  static constexpr int OFF_SCR = (OFF_TMEM + 16 + 1023) / 1024 * 1024;
  static constexpr int ALLOC = OFF_SCR + 8 * ROW_SCRATCH_BYTES + 1024;
  static_assert(ROW_SCRATCH_BYTES % 512 == 0 && ROW_SCRATCH_BYTES >= 2048, "a box per warp");
  static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct DkvBars {
  uint64_t *unit_full, *unit_empty, *kv_full, *kv_empty, *st_full, *st_empty, *s_full, *dp_full, *p_full, *ds_full,
      *acc_full;
};

template <int D>
__device__ __forceinline__ DkvBars dkv_bars(uint8_t* smem) {
  using L = DkvLayout<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  DkvBars r;
  r.unit_full = b;
  r.unit_empty = b + 2;
  r.kv_full = b + 4;
  r.kv_empty = b + 5;
  r.st_full = b + 6;
  r.st_empty = r.st_full + L::STAGES;
  r.s_full = r.st_empty + L::STAGES;  // [2]: one per S^T buffer
  r.dp_full = r.s_full + 2;
  r.p_full = r.s_full + 3;   // [2]: one per 32-column chunk of each warpgroup's half
  r.ds_full = r.s_full + 5;
  r.acc_full = r.s_full + 6;
  return r;
}

struct DkvUnit {
  int b, kvh, kt, q0, nqi, n_it;
  int k0;            // first iteration (block-sparse segment; else 0): iteration k covers
                     // query head kvh * g + (k0 + k) / nqi and query tile (k0 + k) % nqi
  int slot;          // block-sparse split key tile: its partial tile (else -1: write dK, dV)
  const int* qlist;  // block-sparse: the key tile's query tiles (else q0, q0 + 1, ...)
  SeqRows sr;  // the unit's sequence (packed sequences: its own lengths and row offsets)
  bool work;   // the key tile holds keys that some query sees
  bool zero;   // the key tile holds keys that no query sees: their gradients are 0
};

// Key tiles visited by query tile qt: a band's range, else a prefix (causal: up
// to the diagonal tile, Nq == Nk).
template <int MASK>
__device__ __forceinline__ void dq_kv_range(const Dims& s, int qt, int& lo, int& hi) {
  if (MASK == MASK_BAND) {
    kv_range(s, qt, lo, hi);
  } else {
    lo = 0;
    hi = MASK == MASK_CAUSAL ? qt + 1 : k_tiles(s);
  }
}

// The query tiles visiting key tile kt: a band's range, or under j <= i (where
// Nq == Nk) the suffix from the diagonal tile.
template <int MASK, bool VL, bool SP>
__device__ __forceinline__ DkvUnit dkv_decode(const BwdParams& p, int u) {
  const Dims& s = p.dims;
  DkvUnit r;
  r.k0 = 0;
  r.slot = -1;
  int seg_n = 0;
  if (SP) {  // segment-major: unit u = segment u / (B * Hkv) of head group u % (B * Hkv)
    const int heads = s.B * s.Hkv, bh = u % heads;
    const int4 e = __ldg(reinterpret_cast<const int4*>(p.sp_plan + SP_PLAN_SEGS) + u / heads);
    r.b = bh / s.Hkv;
    r.kvh = bh % s.Hkv;
    r.kt = e.x;
    r.k0 = e.y;
    seg_n = e.z;
    r.slot = e.w >= 0 ? bh * __ldg(p.sp_plan + 1) + e.w : -1;
    r.sr = seq_rows<VL>(s, r.b);
  } else if (VL) {  // plan level m = the key tile counted from the sequence's end
    int m;
    plan_unit(p.plan, s.Hkv, u, r.b, r.kvh, m);
    r.sr = seq_rows<VL>(s, r.b);
    r.kt = k_tiles(r.sr.s) - 1 - m;
  } else {
    dkdv_unit(s, u, r.b, r.kvh, r.kt);
    r.sr = seq_rows<VL>(s, r.b);
  }
  const Dims& su = r.sr.s;
  int qhi = q_tiles(su);
  r.qlist = nullptr;
  if (SP) {
    r.q0 = __ldg(p.cols_ptr + r.kt);
    qhi = __ldg(p.cols_ptr + r.kt + 1);
    r.qlist = p.cols_idx + r.q0;
  } else if (MASK == MASK_BAND) {
    q_range(su, r.kt, r.q0, qhi);
  } else {
    r.q0 = MASK == MASK_CAUSAL ? r.kt : 0;
  }
  const bool keys = r.kt < k_tiles(su);
  r.nqi = keys ? imax(0, qhi - r.q0) : 0;
  r.n_it = SP ? seg_n : (s.Hq / s.Hkv) * r.nqi;
  r.work = r.n_it > 0;
  r.zero = keys && !r.work;
  return r;
}

template <int D, int MASK, bool VL, bool SP>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv) {
  using L = DkvLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DkvBars bar = dkv_bars<D>(smem);
  int* unit_slot = reinterpret_cast<int*>(smem + L::OFF_UNIT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const Ctl ctl{p.status, p.timeout_ns};
  const Dims& s = p.dims;
  // units: packed sequences and block-sparse from their plans
  const int total = VL ? __ldg(p.plan) : SP ? __ldg(p.sp_plan) * s.B * s.Hkv : p.total_units;
  const int g = s.Hq / s.Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.unit_full[i], 1);
      mbar_init(&bar.unit_empty[i], 1 + 8);
    }
    mbar_init(bar.kv_full, 1);
    mbar_init(bar.kv_empty, 1);
    for (int i = 0; i < L::STAGES; ++i) {
      mbar_init(&bar.st_full[i], 1);
      mbar_init(&bar.st_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&bar.s_full[i], 1);
    mbar_init(bar.dp_full, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bar.p_full[i], 8);
    mbar_init(bar.ds_full, 8);
    mbar_init(bar.acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the preprocess kernel's statistics (and the cleared header) are complete
  griddep_launch_dependents();  // the dQ kernel may take over SMs as this kernel's CTAs finish

  if (warp == 0) {
    if (lane_id() == 0) {  // ---------------------------------------------- producer
      uint32_t sq = 0, un = 0;  // un: units with work so far (K/V phase)
      int kv_armed = -1;
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&bar.unit_empty[slot], ((it >> 1) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
        const int u = atomicAdd(p.counter, 1);
        unit_slot[slot] = u;
        mbar_arrive(&bar.unit_full[slot]);
        if (u >= total) break;
        const DkvUnit w = dkv_decode<MASK, VL, SP>(p, u);
        if (!w.work) continue;
        const int krow = w.sr.koff + w.kt * TILE, tb = w.sr.tb;
        if (!mbar_wait(bar.kv_empty, (un & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) break;
        mbar_arrive_expect_tx(bar.kv_full, 2 * L::TB);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(smem + L::OFF_K + c * (TILE * 128), &tm_k, bar.kv_full, c * 64, w.kvh, krow, tb);
          tma_load_4d(smem + L::OFF_V + c * (TILE * 128), &tm_v, bar.kv_full, c * 64, w.kvh, krow, tb);
        }
        kv_armed = static_cast<int>(un++);
        bool ok = true;
        for (int k = 0; k < w.n_it; ++k, ++sq) {
          const int st = sq % L::STAGES;
          if (!mbar_wait(&bar.st_empty[st], ((sq / L::STAGES) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) {
            ok = false;
            break;
          }
          const int kk = w.k0 + k;
          const int hq = w.kvh * g + kk / w.nqi, qi = SP ? __ldg(w.qlist + kk % w.nqi) : w.q0 + kk % w.nqi;
          uint8_t* base = smem + L::OFF_ST + st * L::STAGE;
          const int64_t row0 = (static_cast<int64_t>(w.b) * s.Hq + hq) * p.nq_pad + qi * TILE;
          mbar_arrive_expect_tx(&bar.st_full[st], 2 * L::TB + 1024);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(base + c * (TILE * 128), &tm_q, &bar.st_full[st], c * 64, hq, w.sr.qoff + qi * TILE, tb);
            tma_load_4d(base + L::TB + c * (TILE * 128), &tm_do, &bar.st_full[st], c * 64, hq,
                        w.sr.qoff + qi * TILE, tb);
          }
          bulk_load(base + 2 * L::TB, p.neg_lse2 + row0, 512, &bar.st_full[st]);
          bulk_load(base + 2 * L::TB + 512, p.neg_delta + row0, 512, &bar.st_full[st]);
          if (k + 1 < w.n_it) {  // the next iteration's Q and dO into L2 while this stage waits its turn
            const int hq1 = w.kvh * g + (kk + 1) / w.nqi;
            const int qi1 = SP ? __ldg(w.qlist + (kk + 1) % w.nqi) : w.q0 + (kk + 1) % w.nqi;
            for (int c = 0; c < D / 64; ++c) {
              tma_prefetch_l2_4d(&tm_q, c * 64, hq1, w.sr.qoff + qi1 * TILE, tb);
              tma_prefetch_l2_4d(&tm_do, c * 64, hq1, w.sr.qoff + qi1 * TILE, tb);
            }
          }
        }
        if (!ok) break;
      }
      // copies in flight land before exit
      for (int i = 0; i < L::STAGES; ++i)
        if (sq > static_cast<uint32_t>(i)) {
          const uint32_t last = sq - 1 - ((sq - 1 - i) % L::STAGES);
          mbar_wait(&bar.st_full[i], (last / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
        }
      if (kv_armed >= 0) mbar_wait(bar.kv_full, kv_armed & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {  // -------------------------------------------------- MMA issuer
    // The whole warp runs the issue loop converged; one elected lane issues each
    // MMA and commit, so descriptors are formed in uniform registers.
    const uint32_t kb = smem_u32(smem + L::OFF_K), vb = smem_u32(smem + L::OFF_V);
    const uint32_t stb = smem_u32(smem + L::OFF_ST);
    const uint32_t tP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
    auto tS = [&](uint32_t q) { return tmem + ((L::SB == 2 && (q & 1)) ? 384u : 0u); };  // S^T of iteration q
    uint32_t sq = 0, pph = 0, dph = 0, un = 0;
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      if (!warp_wait(&bar.unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
      const int u = unit_slot[slot];
      if (elect_one()) mbar_arrive(&bar.unit_empty[slot]);
      if (u >= total) break;
      const DkvUnit w = dkv_decode<MASK, VL, SP>(p, u);
      if (!w.work) continue;
      if (!warp_wait(bar.kv_full, (un++) & 1, ctl, FA_STATUS_TIMEOUT_MMA)) break;
      bool ok = warp_wait(&bar.st_full[sq % L::STAGES], (sq / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
      if (!ok) break;
      tc_fence_after();
      {
        const uint32_t qb = stb + (sq % L::STAGES) * L::STAGE;
        issue_ss<D, true>(tS(sq), kb, qb);       // S^T = K Q^T
        if (elect_one()) mma_commit(&bar.s_full[sq & (L::SB - 1)]);
        issue_ss<D, true>(tP, vb, qb + L::TB);   // dP^T = V dO^T
        if (elect_one()) {
          mma_commit(bar.dp_full);
          if (w.n_it == 1) mma_commit(bar.kv_empty);  // K and V are read by S and dP only
        }
        if (L::SB == 2 && w.n_it > 1) {  // the second iteration's S^T, into the other buffer
          ok = warp_wait(&bar.st_full[(sq + 1) % L::STAGES], ((sq + 1) / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          issue_ss<D, true>(tS(sq + 1), kb, stb + ((sq + 1) % L::STAGES) * L::STAGE);
          if (elect_one()) mma_commit(&bar.s_full[(sq + 1) & 1]);
        }
      }
      for (int k = 0; k < w.n_it && ok; ++k) {
        const uint32_t cur = stb + ((sq + k) % L::STAGES) * L::STAGE;
        // dV += P^T dO, each half as soon as its P columns are in TMEM
        ok = warp_wait(&bar.p_full[0], pph, ctl, FA_STATUS_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
        issue_ts_half<D, 0, true>(tdV, tS(sq + k), cur + L::TB, k > 0);
        ok = warp_wait(&bar.p_full[1], pph, ctl, FA_STATUS_TIMEOUT_MMA);
        pph ^= 1;
        if (!ok) break;
        tc_fence_after();
        issue_ts_half<D, 1, true>(tdV, tS(sq + k), cur + L::TB, true);
        const bool more = k + 1 < w.n_it;
        const uint32_t nxt = stb + ((sq + k + 1) % L::STAGES) * L::STAGE;  // (used when more)
        if (k + L::SB < w.n_it) {  // S^T of the iteration SB ahead, into the buffer this dV has read
          const uint32_t nsq = sq + k + L::SB;
          ok = warp_wait(&bar.st_full[nsq % L::STAGES], (nsq / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          issue_ss<D, true>(tS(nsq), kb, stb + (nsq % L::STAGES) * L::STAGE);
          if (elect_one()) mma_commit(&bar.s_full[nsq & (L::SB - 1)]);
        }
        // dK += dS^T Q (whole: a second hand-off here costs more than it overlaps)
        ok = warp_wait(bar.ds_full, dph, ctl, FA_STATUS_TIMEOUT_MMA);
        dph ^= 1;
        if (!ok) break;
        tc_fence_after();
        issue_ts_half<D, 0, true>(tdK, tP, cur, k > 0);
        issue_ts_half<D, 1, true>(tdK, tP, cur, true);
        if (elect_one()) mma_commit(&bar.st_empty[(sq + k) % L::STAGES]);
        if (more) {
          issue_ss<D, true>(tP, vb, nxt + L::TB);
          // The unit's last S and dP are issued: K and V can be refilled with the
          // next unit's tiles while its last dV and dK run.
          if (elect_one()) {
            mma_commit(bar.dp_full);
            if (k + 2 == w.n_it) mma_commit(bar.kv_empty);
          }
        }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(bar.acc_full);
      sq += w.n_it;
    }
  } else if (warp >= 4) {  // -------------------------------------------------- gradient warps
    const int wq = warp & 3;
    uint8_t* scratch = smem + L::OFF_SCR + (warp - 4) * ROW_SCRATCH_BYTES;
    const int c0 = ((warp - 4) >> 2) * 64;  // this warpgroup's first column
    const int r = wq * 32 + lane_id();      // key row within the tile
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tP = tmem + lanes + 128, tdV = tmem + lanes + 256, tdK = tmem + lanes + 256 + D;
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t sq = 0, sph[2] = {0, 0}, dph = 0, un = 0;
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      bool ok = mbar_wait(&bar.unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int u = unit_slot[slot];
      warp_arrive(&bar.unit_empty[slot]);
      if (u >= total) break;
      const DkvUnit w = dkv_decode<MASK, VL, SP>(p, u);
      const Dims& su = w.sr.s;  // this unit's sequence
      if (!w.sr.ok && warp == 4 && lane_id() == 0) report(ctl, FA_STATUS_BAD_INPUT);
      if (!w.work) {
        if (w.zero) {  // keys of a sequence without queries: zero gradients, this thread's row and columns
          const int key = w.kt * TILE + r;
          if (key < su.Nk) {
            const int64_t krow = w.sr.koff + static_cast<int64_t>(key);
            uint4* v4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dv.ptr) + w.b * p.dv.sb +
                                                 krow * p.dv.sn + w.kvh * p.dv.sh + (c0 / 64) * (D / 2));
            uint4* k4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dk.ptr) + w.b * p.dk.sb +
                                                 krow * p.dk.sn + w.kvh * p.dk.sh + (c0 / 64) * (D / 2));
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              v4[i] = make_uint4(0, 0, 0, 0);
              k4[i] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        continue;
      }
      const int key = w.kt * TILE + r;
      int qfull_lo = 0, qfull_hi = 0;  // band: query tiles whose rows all see every key of this tile
      if (MASK == MASK_BAND) q_full_range(su, w.kt, qfull_lo, qfull_hi);
      for (int k = 0; k < w.n_it && ok; ++k) {
        const uint32_t q = sq + k;
        const uint8_t* stage = smem + L::OFF_ST + (q % L::STAGES) * L::STAGE;
        const float* nl2 = reinterpret_cast<const float*>(stage + 2 * L::TB);  // -LSE2[query]
        const float* nd = nl2 + 128;                                            // -D[query]
        const int qi = SP ? __ldg(w.qlist + (w.k0 + k) % w.nqi) : w.q0 + k % w.nqi;
        // rows (keys) see only part of the tile's queries: the band's edges, or causal's diagonal
        const bool part = MASK == MASK_BAND ? (qi < qfull_lo || qi > qfull_hi)
                                            : (MASK == MASK_CAUSAL && qi == w.kt);
        const int sb = q & (L::SB - 1);  // this iteration's S^T buffer
        const uint32_t tS = tmem + lanes + (sb ? 384u : 0u);
        ok = mbar_wait(&bar.st_full[q % L::STAGES], (q / L::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
        ok = ok && mbar_wait(&bar.s_full[sb], sph[sb], ctl, FA_STATUS_TIMEOUT_SOFTMAX);
        sph[sb] ^= 1;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P^T[key, query] = exp2(S * scale*log2e - LSE2[query]); causal: 0 where query < key.
        // Elementwise math runs on packed f32x2 operations: scalar FP32 issue at this rate
        // from the other sub-partitions starves the tensor pipe, packed issue does not.
        // This warpgroup's 64 columns of S^T are read at once; P goes back as bf16 over
        // them in two 32-column chunks, each announced on its own barrier so that the
        // dV product starts on the first chunk.  P stays in registers (fp32) for dS.
        float pf[64];
        {
          uint32_t sr[64];
          tmem_ld64(tS + c0, sr);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int e = 32 * cc + 4 * j;
              const float4 l4 = *reinterpret_cast<const float4*>(nl2 + c0 + e);
              const float2 x01 = __ffma2_rn(f32x2(sr[e], sr[e + 1]), c2, make_float2(l4.x, l4.y));
              const float2 x23 = __ffma2_rn(f32x2(sr[e + 2], sr[e + 3]), c2, make_float2(l4.z, l4.w));
              pf[e + 0] = ex2(x01.x);
              pf[e + 1] = ex2(x01.y);
              pf[e + 2] = ex2(x23.x);
              pf[e + 3] = ex2(x23.y);
            }
            if (MASK == MASK_BAND && part) {  // query q sees this key iff key - wr <= q <= key + wl
              const int q_first = qi * TILE + c0 + 32 * cc;
              const int lo = key - s.wr - q_first, hi = key + s.wl + 1 - q_first;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < lo || i >= hi) pf[32 * cc + i] = 0.f;
            } else if (MASK == MASK_CAUSAL && part) {  // columns below lim (queries before this key)
              const int lim = key - qi * TILE - c0 - 32 * cc;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < lim) pf[32 * cc + i] = 0.f;
            }
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(pf[32 * cc + 2 * i], pf[32 * cc + 2 * i + 1]);
            tmem_st16(tS + c0 + 16 * cc, pk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&bar.p_full[cc]);
          }
        }

        ok = mbar_wait(bar.dp_full, dph, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
        dph ^= 1;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dS^T = P^T o (dP^T - D[query]), in the same two chunks, announced together
        {
          uint32_t sr[64];
          tmem_ld64(tP + c0, sr);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t dk[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int e = 32 * cc + 4 * j;
              const float4 d4 = *reinterpret_cast<const float4*>(nd + c0 + e);
              const float2 a = __fmul2_rn(make_float2(pf[e], pf[e + 1]),
                                          __fadd2_rn(f32x2(sr[e], sr[e + 1]), make_float2(d4.x, d4.y)));
              const float2 b = __fmul2_rn(make_float2(pf[e + 2], pf[e + 3]),
                                          __fadd2_rn(f32x2(sr[e + 2], sr[e + 3]), make_float2(d4.z, d4.w)));
              dk[2 * j] = pack_bf16(a.x, a.y);
              dk[2 * j + 1] = pack_bf16(b.x, b.y);
            }
            tmem_st16(tP + c0 + 16 * cc, dk);
            tmem_wait_st();
          }
          tc_fence_before();
          warp_arrive(bar.ds_full);
        }
      }
      if (!ok) break;
      ok = mbar_wait(bar.acc_full, (un++) & 1, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int key0 = w.kt * TILE + wq * 32;  // this warp's first key row (within its sequence)
      const int64_t krow0 = w.sr.koff + static_cast<int64_t>(key0);
      __nv_bfloat16* dv0 = reinterpret_cast<__nv_bfloat16*>(p.dv.ptr) + w.b * p.dv.sb + krow0 * p.dv.sn +
                           w.kvh * p.dv.sh;
      __nv_bfloat16* dk0 = reinterpret_cast<__nv_bfloat16*>(p.dk.ptr) + w.b * p.dk.sb + krow0 * p.dk.sn +
                           w.kvh * p.dk.sh;
      if (SP && w.slot >= 0) {  // a segment of a split key tile: its fp32 partial, row r = [dV | dK]
        float* part = p.sp_pool + (static_cast<int64_t>(w.slot) * TILE + r) * (2 * D) + (c0 / 64) * (D / 2);
        store_acc_f32<D / 2>(tdV, (c0 / 64) * (D / 2), part);
        store_acc_f32<D / 2>(tdK, (c0 / 64) * (D / 2), part + D);
      } else if (!VL && !SP && p.tma_out) {  // dense: 32 x 32 boxes through the copy engine
        if (key0 < su.Nk) {                   // (a warp whose rows all lie past the end stores nothing)
          store_acc_boxes<D / 2>(tdV, (c0 / 64) * (D / 2), 1.f, &tm_dv, w.kvh, key0, w.b, scratch);
          store_acc_boxes<D / 2>(tdK, (c0 / 64) * (D / 2), p.scale, &tm_dk, w.kvh, key0, w.b, scratch);
        }
      } else {
        store_acc_rows<D / 2>(tdV, (c0 / 64) * (D / 2), 1.f, dv0, p.dv.sn, su.Nk - key0, scratch);
        store_acc_rows<D / 2>(tdK, (c0 / 64) * (D / 2), p.scale, dk0, p.dk.sn, su.Nk - key0, scratch);
      }
      sq += w.n_it;
    }
    if (!VL && !SP && p.tma_out && lane_id() == 0) bulk_wait<0>();  // the gradient stores have finished
  }
  // Lanes 1-31 of the producer warp had no role: they wait here for their lane 0,
  // so that every warp reaches the block barrier converged (a barrier met by part
  // of a warp does not hold the rest) and TMEM is freed only after all its users.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The key tiles of dQ unit qt: the range [klo, khi) (dense, band, packed), or
// for block-sparse the query tile's list (klo = 0, khi = its length, *klist).
template <int MASK, bool SP>
__device__ __forceinline__ void dq_keys(const BwdParams& p, const Dims& su, int qt, int& klo, int& khi,
                                        const int*& klist) {
  klist = nullptr;
  if (SP) {
    const int r0 = __ldg(p.rows_ptr + qt);
    klo = 0;
    khi = __ldg(p.rows_ptr + qt + 1) - r0;
    klist = p.rows_idx + r0;
  } else {
    dq_kv_range<MASK>(su, qt, klo, khi);
  }
}

// The dQ unit's (b, h, query tile): dense order, or the packed sequences' plan.
template <bool VL>
__device__ __forceinline__ void dq_unit_of(const BwdParams& p, int u, int& b, int& h, int& qt) {
  if (VL)
    plan_unit(p.plan, p.dims.Hq, u, b, h, qt);
  else
    dq_unit(p.dims, u, b, h, qt);
}

// ================================================================== dQ
template <int D>
struct DqLayout {
  static constexpr int TB = TILE * D * 2;
  // K_j is read by S_j and, two iterations later, by dQ += dS_j K_j; V_j only by dP_j.
  // Separate rings let K run three tiles deep (V two) in the same shared memory.
  static constexpr int KST = D == 64 ? 4 : 3;
  static constexpr int VST = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TB;
  static constexpr int OFF_K = 2 * TB;
  static constexpr int OFF_V = OFF_K + KST * TB;
  static constexpr int OFF_BAR = OFF_V + VST * TB;
  // unit_full[2] unit_empty[2] q_full q_empty k_full[KST] k_empty[KST] v_full[VST] v_empty[VST] s_full[2]
  // dp_full ds_full acc_full
  static constexpr int NBAR = 4 + 2 + 2 * KST + 2 * VST + 5;
  static constexpr int OFF_UNIT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_TMEM = OFF_UNIT + 16;
  static constexpr int OFF_SCR = (OFF_TMEM + 16 + 127) / 128 * 128;  // row-store scratch, one per dQ warp
  // At d = 128 the rings leave no room for a dedicated scratch: the epilogue then
  // stages its rows in the Q tile, which every S of the unit has finished reading,
  // and the dQ warps (not the MMA thread) release Q and dO for the next unit.
  static constexpr bool SCRATCH = OFF_SCR + 8 * ROW_SCRATCH_BYTES + 1024 <= 227 * 1024;
  static_assert(SCRATCH || 8 * ROW_SCRATCH_BYTES <= TB, "the Q tile holds the epilogue scratch");
  static constexpr int ALLOC = (SCRATCH ? OFF_SCR + 8 * ROW_SCRATCH_BYTES : OFF_TMEM + 16) + 1024;
};

template <int D, int MASK, bool VL, bool SP>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using L = DqLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* unit_full = bb;
  uint64_t* unit_empty = bb + 2;
  uint64_t* q_full = bb + 4;
  uint64_t* q_empty = bb + 5;
  uint64_t* k_full = bb + 6;
  uint64_t* k_empty = k_full + L::KST;
  uint64_t* v_full = k_empty + L::KST;
  uint64_t* v_empty = v_full + L::VST;      // arrived by a dQ warp once it has seen dP of that tile done
  uint64_t* s_full = v_empty + L::VST;      // [2]
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_full = s_full + 3;
  uint64_t* acc_full = s_full + 4;
  int* unit_slot = reinterpret_cast<int*>(smem + L::OFF_UNIT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const Ctl ctl{p.status, p.timeout_ns};
  const Dims& s = p.dims;
  const int total = VL ? __ldg(p.plan) : p.total_units;  // units (packed sequences: from the plan)
  const int g = s.Hq / s.Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], 1 + 8);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, L::SCRATCH ? 1 : 8);
    for (int i = 0; i < L::KST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < L::VST; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the preprocess kernel's statistics are complete (dQ launched right after dK/dV: they
  // were before the dK/dV kernel let it start, and dQ reads nothing dK/dV writes)
  if (!p.dq_after_dkdv) griddep_wait();

  if (warp == 0) {
    if (lane_id() == 0) {  // ---------------------------------------------- producer
      uint32_t kq = 0, qn = 0;  // qn: units with work so far (Q phase)
      int q_armed = -1;
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&unit_empty[slot], ((it >> 1) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
        const int u = atomicAdd(p.counter, 1);
        unit_slot[slot] = u;
        mbar_arrive(&unit_full[slot]);
        if (u >= total) break;
        int b, h, qt;
        dq_unit_of<VL>(p, u, b, h, qt);
        const SeqRows sr = seq_rows<VL>(s, b);
        if (qt >= q_tiles(sr.s)) continue;  // past its (packed) sequence
        int klo, khi;
        const int* klist;
        dq_keys<MASK, SP>(p, sr.s, qt, klo, khi, klist);
        const int n = khi - klo, kvh = h / g;
        if (SP && n == 0) continue;  // no key tile listed: the dQ warps write zeros
        if (!mbar_wait(q_empty, (qn & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) break;
        mbar_arrive_expect_tx(q_full, 2 * L::TB);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(smem + L::OFF_Q + c * (TILE * 128), &tm_q, q_full, c * 64, h, sr.qoff + qt * TILE, sr.tb);
          tma_load_4d(smem + L::OFF_DO + c * (TILE * 128), &tm_do, q_full, c * 64, h, sr.qoff + qt * TILE, sr.tb);
        }
        q_armed = static_cast<int>(qn++);
        bool ok = true;
        for (int j = 0; j < n; ++j, ++kq) {
          // K_j: its slot is free once dQ of the tile KST back is done.
          const int ks = kq % L::KST;
          if (!mbar_wait(&k_empty[ks], ((kq / L::KST) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[ks], L::TB);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(smem + L::OFF_K + ks * L::TB + c * (TILE * 128), &tm_k, &k_full[ks], c * 64, kvh,
                        sr.koff + (SP ? __ldg(klist + j) : klo + j) * TILE, sr.tb);
          // V_j: its slot is free once dP of the tile VST back is done.
          const int vs = kq % L::VST;
          if (!mbar_wait(&v_empty[vs], ((kq / L::VST) & 1) ^ 1, ctl, FA_STATUS_TIMEOUT_LOAD)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[vs], L::TB);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(smem + L::OFF_V + vs * L::TB + c * (TILE * 128), &tm_v, &v_full[vs], c * 64, kvh,
                        sr.koff + (SP ? __ldg(klist + j) : klo + j) * TILE, sr.tb);
        }
        if (!ok) break;
      }
      // copies in flight land before exit (v_full of a slot may trail its k_full by one load)
      for (int i = 0; i < L::KST; ++i)
        if (kq > static_cast<uint32_t>(i)) {
          const uint32_t last = kq - 1 - ((kq - 1 - i) % L::KST);
          mbar_wait(&k_full[i], (last / L::KST) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
        }
      for (int i = 0; i < L::VST; ++i)
        if (kq > static_cast<uint32_t>(i)) {
          const uint32_t last = kq - 1 - ((kq - 1 - i) % L::VST);
          mbar_wait(&v_full[i], (last / L::VST) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
        }
      if (q_armed >= 0) mbar_wait(q_full, q_armed & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {  // -------------------------------------------------- MMA issuer
    // The whole warp runs the issue loop converged; one elected lane issues each
    // MMA and commit, so descriptors are formed in uniform registers.
    const uint32_t qb = smem_u32(smem + L::OFF_Q), dob = smem_u32(smem + L::OFF_DO);
    const uint32_t kb0 = smem_u32(smem + L::OFF_K), vb0 = smem_u32(smem + L::OFF_V);
    const uint32_t tP = tmem + 256, tdQ = tmem + 384;
    uint32_t kq = 0, dsph = 0, qn = 0;
    auto kwait = [&](uint32_t idx) {
      return warp_wait(&k_full[idx % L::KST], (idx / L::KST) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
    };
    auto vwait = [&](uint32_t idx) {
      return warp_wait(&v_full[idx % L::VST], (idx / L::VST) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
    };
    auto kbase = [&](uint32_t idx) { return kb0 + (idx % L::KST) * L::TB; };
    auto vbase = [&](uint32_t idx) { return vb0 + (idx % L::VST) * L::TB; };
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      if (!warp_wait(&unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT)) break;
      const int u = unit_slot[slot];
      if (elect_one()) mbar_arrive(&unit_empty[slot]);
      if (u >= total) break;
      int b, h, qt;
      dq_unit_of<VL>(p, u, b, h, qt);
      const Dims su = seq_rows<VL>(s, b).s;
      if (qt >= q_tiles(su)) continue;  // past its (packed) sequence
      int klo, khi;
      const int* klist;
      dq_keys<MASK, SP>(p, su, qt, klo, khi, klist);
      const int n = khi - klo;
      if (SP && n == 0) continue;
      bool ok = warp_wait(q_full, (qn++) & 1, ctl, FA_STATUS_TIMEOUT_MMA);
      ok = ok && kwait(kq);
      if (!ok) break;
      tc_fence_after();
      issue_ss<D, true>(tmem + 0, qb, kbase(kq));            // S_0 = Q K_0^T
      if (elect_one()) mma_commit(&s_full[0]);
      if (!vwait(kq)) break;
      tc_fence_after();
      issue_ss<D, true>(tP, dob, vbase(kq));                  // dP_0 = dO V_0^T
      if (elect_one()) mma_commit(dp_full);
      if (n > 1) {
        if (!kwait(kq + 1)) break;
        tc_fence_after();
        issue_ss<D, true>(tmem + 128, qb, kbase(kq + 1));
        if (elect_one()) mma_commit(&s_full[1]);
      }
      for (int j = 0; j < n && ok; ++j) {
        ok = warp_wait(ds_full, dsph, ctl, FA_STATUS_TIMEOUT_MMA);
        dsph ^= 1;
        if (!ok) break;
        tc_fence_after();
        issue_ts<D, true>(tdQ, tP, kbase(kq + j), j > 0);       // dQ += dS K_j
        if (elect_one()) mma_commit(&k_empty[(kq + j) % L::KST]);
        if (j + 1 < n) {
          ok = vwait(kq + j + 1);
          if (!ok) break;
          tc_fence_after();
          issue_ss<D, true>(tP, dob, vbase(kq + j + 1));          // dP_{j+1}
          if (elect_one()) mma_commit(dp_full);
        }
        if (j + 2 < n) {
          ok = kwait(kq + j + 2);
          if (!ok) break;
          tc_fence_after();
          issue_ss<D, true>(tmem + (j & 1) * 128, qb, kbase(kq + j + 2));
          if (elect_one()) mma_commit(&s_full[j & 1]);
        }
      }
      if (!ok) break;
      if (elect_one()) {
        mma_commit(acc_full);
        if (L::SCRATCH) mma_commit(q_empty);
      }
      kq += n;
    }
  } else if (warp >= 4) {  // -------------------------------------------------- gradient warps
    const int wq = warp & 3;
    uint8_t* scratch = smem + (L::SCRATCH ? L::OFF_SCR : L::OFF_Q) + (warp - 4) * ROW_SCRATCH_BYTES;
    const int c0 = ((warp - 4) >> 2) * 64;  // this warpgroup's first key column
    const int r = wq * 32 + lane_id();
    const uint32_t lanes = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tP = tmem + lanes + 256, tdQ = tmem + lanes + 384;
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t sph[2] = {0, 0}, dph = 0, kq = 0, qn = 0;
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      bool ok = mbar_wait(&unit_full[slot], (it >> 1) & 1, ctl, FA_STATUS_TIMEOUT_UNIT);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int u = unit_slot[slot];
      warp_arrive(&unit_empty[slot]);
      if (u >= total) break;
      int b, h, qt;
      dq_unit_of<VL>(p, u, b, h, qt);
      const SeqRows sr = seq_rows<VL>(s, b);
      if (!sr.ok && warp == 4 && lane_id() == 0) report(ctl, FA_STATUS_BAD_INPUT);
      const Dims& su = sr.s;  // this unit's sequence
      if (qt >= q_tiles(su)) continue;  // past its (packed) sequence
      int klo, khi, full_lo = 0, full_hi = 0;
      const int* klist;
      dq_keys<MASK, SP>(p, su, qt, klo, khi, klist);
      if (MASK == MASK_BAND) {
        kv_full_range(su, qt, full_lo, full_hi);
        if ((su.Nk % TILE) != 0) full_hi = imin(full_hi, k_tiles(su) - 2);  // the ragged last tile is masked too
      }
      const int n = khi - klo;
      const int q_row = qt * TILE + r;
      if (SP && n == 0) {  // no key tile listed: dQ = 0 for the tile's rows (this warp's half of the columns)
        if (q_row < su.Nq) {
          uint4* z = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq.ptr) + b * p.dq.sb +
                                              static_cast<int64_t>(q_row) * p.dq.sn + h * p.dq.sh + (c0 / 64) * (D / 2));
#pragma unroll
          for (int i = 0; i < D / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int64_t srow = (static_cast<int64_t>(b) * s.Hq + h) * p.nq_pad + q_row;
      const float2 nl2 = make_float2(p.neg_lse2[srow], p.neg_lse2[srow]);
      const float2 nd2 = make_float2(p.neg_delta[srow], p.neg_delta[srow]);
      for (int j = 0; j < n && ok; ++j) {
        const int bi = j & 1;
        ok = mbar_wait(&s_full[bi], sph[bi], ctl, FA_STATUS_TIMEOUT_SOFTMAX);
        sph[bi] ^= 1;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P = exp2(S * scale*log2e - LSE2[row]), on packed f32x2 operations (see the
        // dK/dV kernel); keys outside the row's band, or past Nk, are masked.
        float pf[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[32];
          tmem_ld32(tmem + lanes + bi * 128 + c0 + 32 * cc, sr);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = __ffma2_rn(f32x2(sr[2 * i], sr[2 * i + 1]), c2, nl2);
            pf[32 * cc + 2 * i] = ex2(x.x);
            pf[32 * cc + 2 * i + 1] = ex2(x.y);
          }
        }
        if (MASK == MASK_BAND) {
          const int kt = klo + j;
          if (kt < full_lo || kt > full_hi) {
            // visible keys [lo, hi) relative to this warpgroup's first column
            const int first = kt * TILE + c0;
            const int hi = imin(su.Nk, q_row + s.wr + 1) - first;
            const int lo = q_row - s.wl - first;
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i < lo || i >= hi) pf[i] = 0.f;
          }
        } else if (SP) {  // the listed tile: the diagonal, or the ragged last tile, is masked
          const int kt = __ldg(klist + j);
          if ((MASK == MASK_CAUSAL && kt == qt) || (kt == k_tiles(su) - 1 && (su.Nk % TILE) != 0)) {
            int lim = imin(TILE, su.Nk - kt * TILE);
            if (MASK == MASK_CAUSAL) lim = imin(lim, q_row - kt * TILE + 1);
            lim -= c0;
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i >= lim) pf[i] = 0.f;
          }
        } else if (j == n - 1) {  // causal or full: only the last key tile holds masked keys
          int lim = imin(TILE, su.Nk - j * TILE);
          if (MASK == MASK_CAUSAL) lim = imin(lim, q_row - j * TILE + 1);
          lim -= c0;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim) pf[i] = 0.f;
        }
        ok = mbar_wait(dp_full, dph, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
        dph ^= 1;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (warp == 4 && lane_id() == 0) mbar_arrive(&v_empty[(kq + j) % L::VST]);  // dP_j done: V_j is free
        tc_fence_after();
        // dS = P o (dP - D_row), written as bf16 over the dP columns already read
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[32];
          tmem_ld32(tP + c0 + 32 * cc, sr);
          uint32_t ds[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 g = __fmul2_rn(make_float2(pf[32 * cc + 2 * i], pf[32 * cc + 2 * i + 1]),
                                        __fadd2_rn(f32x2(sr[2 * i], sr[2 * i + 1]), nd2));
            ds[i] = pack_bf16(g.x, g.y);
          }
          tmem_st16(tP + c0 + 16 * cc, ds);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(ds_full);
      }
      if (!ok) break;
      ok = mbar_wait(acc_full, (qn++) & 1, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int q0 = qt * TILE + wq * 32;  // this warp's first query row (within its sequence)
      __nv_bfloat16* dq0 = reinterpret_cast<__nv_bfloat16*>(p.dq.ptr) + b * p.dq.sb +
                           (sr.qoff + static_cast<int64_t>(q0)) * p.dq.sn + h * p.dq.sh;
      store_acc_rows<D / 2>(tdQ, (c0 / 64) * (D / 2), p.scale, dq0, p.dq.sn, su.Nq - q0, scratch);
      if (!L::SCRATCH) {  // the Q tile was the scratch: order these accesses before the next TMA write
        fence_proxy_async_smem();
        warp_arrive(q_empty);
      }
      kq += n;
    }
  }
  // Lanes 1-31 of the producer warp had no role: they wait here for their lane 0,
  // so that every warp reaches the block barrier converged (a barrier met by part
  // of a warp does not hold the rest) and TMEM is freed only after all its users.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================== block-sparse reduce
// dK, dV of the split key tiles: each output element is the sum of its tile's
// partials in segment order (a fixed order: deterministic), dK times the scale.
// One float4 of a partial row per thread and step; grid-stride.
template <int D>
__global__ void __launch_bounds__(256) bwd_sparse_reduce_kernel(const BwdParams p) {
  const Dims& s = p.dims;
  const int sph = __ldg(p.sp_plan + 1), nsplit = __ldg(p.sp_plan + 2);
  constexpr int ROW4 = 2 * D / 4;          // float4s per partial row
  constexpr int TILE4 = TILE * ROW4;       // ... per partial tile
  const int64_t total = static_cast<int64_t>(s.B) * s.Hkv * nsplit * TILE4;
  const float4* pool = reinterpret_cast<const float4*>(p.sp_pool);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % TILE4);
    const int64_t t = i / TILE4;
    const int j = static_cast<int>(t % nsplit), bh = static_cast<int>(t / nsplit);
    const int4 e = __ldg(reinterpret_cast<const int4*>(p.sp_plan + SP_PLAN_SPLITS) + j);
    const int row = c / ROW4, col = (c % ROW4) * 4;
    const int key = e.x * TILE + row;
    if (key >= s.Nk) continue;
    const float4* src = pool + (static_cast<int64_t>(bh) * sph + e.y) * TILE4 + c;
    float4 a = __ldg(src);
    for (int k = 1; k < e.z; ++k) {
      const float4 x = __ldg(src + static_cast<int64_t>(k) * TILE4);
      a.x += x.x;
      a.y += x.y;
      a.z += x.z;
      a.w += x.w;
    }
    const int b = bh / s.Hkv, kvh = bh % s.Hkv;
    const OutRows& o = col < D ? p.dv : p.dk;
    const float m = col < D ? 1.f : p.scale;
    const float2 lo = __fmul2_rn(make_float2(a.x, a.y), make_float2(m, m));
    const float2 hi = __fmul2_rn(make_float2(a.z, a.w), make_float2(m, m));
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(o.ptr) + b * o.sb + static_cast<int64_t>(key) * o.sn +
                         kvh * o.sh + (col < D ? col : col - D);
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(lo.x, lo.y), pack_bf16(hi.x, hi.y));
  }
}

// Launch with programmatic stream serialisation: the kernel may start while the one
// before it in the stream finishes (it waits with griddepcontrol before depending on it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, int MASK, bool VL = false, bool SP = false>
cudaError_t launch_bwd_t(const BwdLaunch& a, cudaStream_t st) {
  BwdParams p;
  p.plan = nullptr;
  p.tma_out = 0;
  p.dq_after_dkdv = 0;
  p.rows_ptr = a.rows_ptr;
  p.rows_idx = a.rows_idx;
  p.cols_ptr = a.cols_ptr;
  p.cols_idx = a.cols_idx;
  p.sp_plan = a.sp_plan;
  p.sp_pool = a.sp_pool;
  p.dims = a.dims;
  p.scale = a.scale;
  p.scale_log2 = a.scale * LOG2E;
  p.o = a.o;
  p.o_res = a.o_res;
  p.dout = a.dout;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.lse = a.lse;
  p.neg_lse2 = a.neg_lse2;
  p.neg_delta = a.neg_delta;
  p.nq_pad = a.nq_pad;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  // 0) packed sequences: the dQ plan (the query tiles that exist) serves preprocess and dQ
  if (VL && (a.parts & 5)) {
    cudaError_t e = launch_varlen_plan(a.dims, VARLEN_PLAN_DQ, q_tiles(a.dims), a.dims.Hq, a.plan_dq, a.status, st);
    if (e != cudaSuccess) return e;
  }
  // 1) preprocess
  if (a.parts & 1) {
    if (VL) {
      // units <= Hq x (query tiles of all sequences) <= Hq x (total_q / 128 + B)
      const int64_t units = static_cast<int64_t>(a.dims.Hq) * (cdiv(a.dims.total_q, TILE) + a.dims.B);
      const int64_t blocks = units * (TILE / (256 / (D / 8)));
      if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
      bwd_preprocess_varlen_kernel<D><<<static_cast<unsigned>(imax(1, static_cast<int>(blocks))), 256, 0, st>>>(
          p, a.plan_dq);
    } else {
      const int64_t threads = static_cast<int64_t>(a.dims.B) * a.dims.Hq * a.nq_pad * (D / 8);
      cudaError_t e = launch_pdl(bwd_preprocess_kernel<D>, static_cast<unsigned>((threads + 255) / 256), 256, 0, st, p);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2) dK / dV
  if (a.parts & 2) {
    auto kern = bwd_dkdv_kernel<D, MASK, VL, SP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvLayout<D>::ALLOC);
    if (e != cudaSuccess) return e;
    p.counter = a.counters;
    p.total_units = dkdv_units(a.dims);
    p.plan = a.plan_dkdv;
    if (VL) {
      e = launch_varlen_plan(a.dims, VARLEN_PLAN_DKDV, k_tiles(a.dims), a.dims.Hkv, a.plan_dkdv, a.status, st);
      if (e != cudaSuccess) return e;
    }
    // block-sparse: the unit count is on the device; fill the GPU and let the plan's count stop the CTAs
    const int grid = SP ? a.num_sms : imax(1, imin(p.total_units, a.num_sms));
    p.tma_out = (!VL && !SP) ? a.tma_out : 0;
    if (!VL && !SP) {
      e = launch_pdl(kern, grid, 384, DkvLayout<D>::ALLOC, st, a.tm_q, a.tm_k, a.tm_v, a.tm_do, p, a.tm_dk, a.tm_dv);
      if (e != cudaSuccess) return e;
    } else {
      kern<<<grid, 384, DkvLayout<D>::ALLOC, st>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, p, a.tm_dk, a.tm_dv);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (SP) {
      bwd_sparse_reduce_kernel<D><<<2 * a.num_sms, 256, 0, st>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  // 3) dQ
  if (a.parts & 4) {
    auto kern = bwd_dq_kernel<D, MASK, VL, SP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<D>::ALLOC);
    if (e != cudaSuccess) return e;
    p.counter = a.counters + 1;
    p.total_units = dq_units(a.dims);
    p.plan = a.plan_dq;  // built above
    p.dq_after_dkdv = (!VL && !SP && (a.parts & 2)) ? 1 : 0;
    if (!VL && !SP) {
      e = launch_pdl(kern, imax(1, imin(p.total_units, a.num_sms)), 384, DqLayout<D>::ALLOC, st, a.tm_q, a.tm_k,
                     a.tm_v, a.tm_do, p);
      if (e != cudaSuccess) return e;
    } else {
      kern<<<imax(1, imin(p.total_units, a.num_sms)), 384, DqLayout<D>::ALLOC, st>>>(a.tm_q, a.tm_k, a.tm_v,
                                                                                     a.tm_do, p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st) {
  const int m = mask_kind(a.dims);
  if (a.rows_ptr != nullptr) {  // block-sparse: dense batch, no band
    if (a.dims.cu_q != nullptr || m == MASK_BAND) return cudaErrorInvalidValue;
    if (a.d == 64)
      return m == MASK_CAUSAL ? launch_bwd_t<64, MASK_CAUSAL, false, true>(a, st)
                              : launch_bwd_t<64, MASK_NONE, false, true>(a, st);
    return m == MASK_CAUSAL ? launch_bwd_t<128, MASK_CAUSAL, false, true>(a, st)
                            : launch_bwd_t<128, MASK_NONE, false, true>(a, st);
  }
  if (a.dims.cu_q != nullptr) {  // packed sequences: no band
    if (m == MASK_BAND) return cudaErrorInvalidValue;
    if (a.d == 64)
      return m == MASK_CAUSAL ? launch_bwd_t<64, MASK_CAUSAL, true>(a, st) : launch_bwd_t<64, MASK_NONE, true>(a, st);
    return m == MASK_CAUSAL ? launch_bwd_t<128, MASK_CAUSAL, true>(a, st) : launch_bwd_t<128, MASK_NONE, true>(a, st);
  }
  if (a.d == 64)
    return m == MASK_BAND ? launch_bwd_t<64, MASK_BAND>(a, st)
           : m == MASK_CAUSAL ? launch_bwd_t<64, MASK_CAUSAL>(a, st) : launch_bwd_t<64, MASK_NONE>(a, st);
  return m == MASK_BAND ? launch_bwd_t<128, MASK_BAND>(a, st)
         : m == MASK_CAUSAL ? launch_bwd_t<128, MASK_CAUSAL>(a, st) : launch_bwd_t<128, MASK_NONE>(a, st);
}

}  // namespace fa
