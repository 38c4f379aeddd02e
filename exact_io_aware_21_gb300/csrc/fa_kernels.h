// Launch interfaces between the C-ABI layer (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_plan.h"

namespace fa {

struct OutRows {           // a bf16 [B, N, H, d] tensor written row by row
  void* ptr;
  int64_t sb, sn, sh;
};

// Static schedule of the causal forward: the work units of each CTA, balanced on the
// host (fa_sched.cu).  Units of a causal forward differ in cost by up to 20x, and the
// longest-first order handed out dynamically still leaves the last CTAs idle for about
// one small unit; a balanced assignment computed once per shape closes most of that.
// on = 0: units are claimed dynamically (an atomic counter), longest first.
constexpr int SCHED_MAX_CTAS = 160;
constexpr int SCHED_MAX_UNITS = 2048;
struct FwdSched {
  int on;
  int grid;                              // the launch's CTAs (the plan is for exactly this grid)
  uint16_t start[SCHED_MAX_CTAS + 1];    // CTA c runs ord[start[c] .. start[c + 1]) in order
  uint16_t ord[SCHED_MAX_UNITS];
};
// The balanced schedule of a dense causal forward on `grid` CTAs, or nullptr (not
// causal, packed, too many units or CTAs).  Cached per shape; thread-safe.
const FwdSched* causal_schedule(const Dims& s, int d, bool fp8, int grid);

struct FwdLaunch {
  Dims dims;
  int d;
  float scale;
  float tau;  // conditional rescaling: the reference max moves only past this margin (log2 units)
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps, box 64 x 1 x 128 x 1, 128B swizzle
  // output maps for TMA stores (dense bf16 forward): box 32 x 1 x 32 x 1, 64B swizzle
  CUtensorMap tm_o, tm_r;
  int tma_out;      // 1: O (and its residual) leave through tm_o / tm_r
  OutRows o;
  OutRows o_res;   // ptr == nullptr: residual not written
  float* lse;
  int* status;
  int* counter;
  unsigned long long timeout_ns;
  int num_sms;
  // E4M3 operands (sq != nullptr; maps over one-byte codes, box 128 x 1 x 128 x 1):
  // Q block scales [B, Hq, ceil(Nq/128)], K block scales [B, Hkv, ceil(Nk/128)],
  // V scales [B, Hkv]
  const float* sq;
  const float* sk;
  const float* sv;
  // block-sparse (row_ptr != nullptr): CSR table of key tiles per query tile
  const int* row_ptr;  // [ceil(Nq/128) + 1]
  const int* col_idx;  // [nnz]
  int nnz;
  int* plan;           // packed sequences: workspace for the device-side work plan
  unsigned long long* trace;  // timestamps (diag == DG_TRACE); layout below
  int diag;                   // DG_NONE, or a diagnostic instantiation (below)
  const FwdSched* sched;      // static schedule (causal), or nullptr: dynamic claims
  // key-split units (dense bf16 forward without a mask, nsplit > 1): units from
  // split0 on run as nsplit parts along the keys, each writing its O (normalised
  // by its own sum, fp32 [part][2 tiles][128 rows][d]) and LSE ([part][2][128])
  // to part_o / part_lse; a combine kernel then writes O, its residual and LSE
  int split0, nsplit;
  float* part_o;
  float* part_lse;
};
// The key-split plan of a forward (dense, bf16, no mask, no block-sparse table):
// the units of the last, partial wave of SMs (all units when there are fewer
// than SMs) split into nsplit parts of whole key tiles.  nsplit = 1: none.
struct FwdSplit {
  int split0, nsplit;
};
FwdSplit fwd_split_plan(const Dims& s, int sms);
// Diagnostic instantiations of the dense bf16 d = 128 forward: DG_TRACE writes
// timestamps into `trace`; DG_WITHHOLD (tests of the bounded waits) has one softmax
// warp of work unit 0 skip its first P hand-off, so that CTA's MMA issuer's wait runs out.
constexpr int DG_NONE = 0, DG_TRACE = 1, DG_WITHHOLD = 2;
// Zero a workspace header; a forward launched next may start its set-up meanwhile.
cudaError_t launch_header_clear(void* ws, cudaStream_t st);
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t st);

// Forward trace (diagnostics), %globaltimer nanoseconds.  Per CTA c < TRACE_MAX_CTAS:
// [4c] start (after set-up), [4c+1] end (its last role's exit), [4c+2] SM id,
// [4c+3] units run.  Per work
// unit u: [TRACE_UNIT0 + 16u + k], k = 0 claimed, 1 first product issued, 2 last
// product issued, 3 output written (the later query tile), 4 CTA; per query tile t
// of the unit (softmax warps): 5 + t its first S received, 7 + t its last P handed
// over, 9 + t its final O ready (products done), 11 + t its output written.
constexpr int TRACE_MAX_CTAS = 1024;
constexpr int TRACE_UNIT0 = 4 * TRACE_MAX_CTAS;
constexpr int TRACE_UNIT_WORDS = 16;

struct BwdLaunch {
  Dims dims;
  int d;
  float scale;
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  OutRows o, o_res, dout, dq, dk, dv;  // o_res.ptr may be nullptr
  const float* lse;
  float* neg_lse2;   // workspace [B*Hq, Nq_pad] : -LSE * log2(e)  (-inf in padding)
  float* neg_delta;  // workspace [B*Hq, Nq_pad] : -D, D = rowsum(dO o O)
  int nq_pad;
  int* status;
  int* counters;   // [2]
  unsigned long long timeout_ns;
  int num_sms;
  int parts;       // bit 0: preprocess, bit 1: dK/dV, bit 2: dQ
  int* plan_dkdv;  // packed sequences: workspace for the device-side work plans
  int* plan_dq;
  // block-sparse (rows_ptr != nullptr): filtered lists and the dK/dV plan (see SparseLaunch)
  const int* rows_ptr;
  const int* rows_idx;
  const int* cols_ptr;
  const int* cols_idx;
  const int* sp_plan;
  float* sp_pool;  // partial tiles of split key tiles
  // dense bf16 (tma_out = 1): dK and dV leave through TMA stores (maps as the forward's output)
  CUtensorMap tm_dk, tm_dv;
  int tma_out;
};
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st);

struct DecodeLaunch {
  Dims dims;       // causal = 0
  int d;
  float scale;
  CUtensorMap tm_k, tm_v;
  const void* q;
  int64_t q_sb, q_sn, q_sh;
  OutRows o;
  float* lse;
  float* lse_part;  // [B, Hq, Nq, S]
  float* o_part;    // [B, Hq, Nq, S, d]
  int num_splits;
  int chunk;        // keys per split (multiple of 128); paged: computed per sequence in the kernel
  int* status;
  unsigned long long timeout_ns;
  // paged, variable-length cache (block_table == nullptr: contiguous [B, Nk, Hkv, d])
  const int* block_table;  // [B, max_pages] physical page of each logical page
  int max_pages;
  const int* seqlens;      // [B] keys of each sequence, 1..Nk
  int num_pages;
  int page_size;           // 16, 32, 64, or a multiple of 128
  // paged head groups: K/V heads per CTA (8, 4 or 2; 0 = one head per CTA).  A stage
  // holds 128 / head_group keys of each head; tm_k / tm_v then map (channel, row,
  // head, page) with boxes of 64 x min(page_size, 128 / head_group) x head_group
  int head_group;
};
constexpr int DECODE_HEAD_GROUP = 8;  // the largest head group
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t st);

struct QuantLaunch {       // E4M3 codes of a bf16 [B, N, H, d] tensor
  const void* x;
  int64_t sb, sn, sh;      // x strides (elements)
  int B, N, H, d;
  const float* signs;      // d signs of the Hadamard rotation, or nullptr
  void* out;               // uint8 [B, N, H, d]
  int64_t ob, on, oh;      // out strides (bytes)
  float* scales;           // per_block: [B, H, nblk]; else [B, H]
  unsigned* head_amax;     // per-head pass: [B, H] zeroed workspace
  int nblk;                // ceil(N / 128)
  int per_block;
  CUtensorMap tm_x;        // x as 4-D map, box 64 x 1 x 128 x 1, 128-byte swizzle
  int* status;             // workspace status word (a wait that ran out)
  unsigned long long timeout_ns;
  int num_sms;
};
cudaError_t launch_quantize(const QuantLaunch& a, cudaStream_t st);

// Block-sparse backward: the caller's CSR table checked and filtered into
// per-query-tile and per-key-tile lists (ascending), via a tile bitmap in
// shared memory, and the dK/dV segment plan built from the lists' lengths.
struct SparseLaunch {
  const int* row_ptr;   // caller's table: [nqt + 1], col_idx [nnz]
  const int* col_idx;
  int nnz, nqt, nkt, causal;
  int group;            // query heads per K/V head
  int heads;            // B * Hkv: copies of the dK/dV plan's segments
  int pool_slots;       // partial tiles the workspace holds (all heads)
  int* rows_ptr;        // out [nqt + 1], rows_idx [<= nnz]: key tiles of each query tile
  int* rows_idx;
  int* cols_ptr;        // out [nkt + 1], cols_idx [<= nnz]: query tiles of each key tile
  int* cols_idx;
  int* dkdv_plan;       // out [SP_PLAN_INTS]: the dK/dV segment plan (layout below)
  int* status;
};
cudaError_t launch_sparse_lists(const SparseLaunch& a, cudaStream_t st);

// Block-sparse dK/dV segment plan.  A key tile's iterations (query heads of the
// group x its listed query tiles, flattened) form one unit, or, when there are
// more than `seg` of them, near-equal segments of at most `seg`; each segment
// of a split tile owns a partial tile (fp32 dV | dK, [128][2d]) that a reduce
// kernel sums in segment order.  The segments of one head group are ordered
// longest first and repeated for every (batch, K/V head).
//   [0] segments per head group  [1] partial slots per head group
//   [2] split key tiles          [3] seg
//   SP_PLAN_SEGS + 4 i: segment i = {key tile, first iteration, iterations, slot or -1}
//   SP_PLAN_SPLITS + 4 j: split tile j = {key tile, first slot, segments, 0}
constexpr int SP_PLAN_PARALLELISM = 152;  // the units' target: one GB300's SMs (the plan is device-independent)
constexpr int SP_MIN_SEGMENT = 32;
constexpr int SP_MAX_SEGMENTS = 1024 + 2 * SP_PLAN_PARALLELISM;
constexpr int SP_PLAN_SEGS = 4;
constexpr int SP_PLAN_SPLITS = SP_PLAN_SEGS + 4 * SP_MAX_SEGMENTS;
constexpr int SP_PLAN_INTS = SP_PLAN_SPLITS + 4 * 1024;

// Device-side work plan of packed sequences (levels: forward pairs, dQ query
// tiles, dK/dV key tiles from the end); `plan` holds varlen_plan_ints(nlev, B) ints.
constexpr int VARLEN_PLAN_FWD = 0, VARLEN_PLAN_DQ = 1, VARLEN_PLAN_DKDV = 2;
// Sequences the cu arrays cannot hold are reported in *status and get no units.
cudaError_t launch_varlen_plan(const Dims& d, int mode, int nlev, int heads, int* plan, int* status,
                               cudaStream_t st);

cudaError_t launch_selftest_mma(int mode, int n_or_k, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const void* a_rows, float* c, int* status, cudaStream_t st);

}  // namespace fa
