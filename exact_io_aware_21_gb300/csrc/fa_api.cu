// C ABI of libfa_gb300.so (declared in include/fa.h): argument checks, TMA
// descriptor encoding, workspace layout, and the launches.  No allocation, no
// synchronisation and no host-side compute fallback: every attention result
// comes from the kernels in fa_fwd.cu, fa_bwd.cu and fa_decode.cu.
#include <math.h>
#include <string.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_kernels.h"
#include "fa_plan.h"
#include "fa_status.h"

using namespace fa;

namespace {

unsigned long long g_timeout_ns = 10ull * 1000 * 1000 * 1000;
int g_last_cuda_error = 0;
void* g_trace = nullptr;  // forward timestamps (fa_set_trace)
size_t g_trace_bytes = 0;
bool g_withhold = false;  // the next dense d = 128 forward runs the withheld-hand-off test kernel

int cuda_fail(cudaError_t e, int code) {
  g_last_cuda_error = static_cast<int>(e);
  return code;
}

// ---- device facts ---------------------------------------------------------------
struct DevInfo {
  int ok = -1;  // -1 unknown, 0 not sm_103, 1 sm_103
  int sms = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

int device_info(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_CUDA);
  if (dev < 0 || dev >= 64) return FA_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, FA_ERR_CUDA);
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
  }
  if (d.ok != 1) return FA_ERR_ARCH;
  *sms = d.sms;
  return FA_OK;
}

// ---- TMA descriptor encoding ------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D map over a bf16 [B, N, H, d] tensor: dims (d, H, N, B); box 64 x 1 x 128 x 1,
// 128-byte swizzle; rows past N read as zero.
int make_map(CUtensorMap* m, const void* ptr, int B, int N, int H, int d, int64_t sb, int64_t sn, int64_t sh,
             int box_rows = TILE) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(sn) * 2,
                           static_cast<cuuint64_t>(sb) * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ALIGN;
}

// Map for TMA stores of a bf16 [B, N, H, d] output: boxes of 32 channels x 32 rows
// (one warp's rows, 64 bytes each), 64-byte swizzle; rows past N are dropped.
int make_store_map(CUtensorMap* m, const void* ptr, int B, int N, int H, int d, int64_t sb, int64_t sn, int64_t sh) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(sn) * 2,
                           static_cast<cuuint64_t>(sb) * 2};
  cuuint32_t box[4] = {32, 1, 32, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ALIGN;
}

// The same map over one-byte elements (E4M3 codes): box 128 x 1 x box_rows x 1,
// the 128-byte inner box matching the 128-byte swizzle.  Strides in elements.
int make_map_u8(CUtensorMap* m, const void* ptr, int B, int N, int H, int d, int64_t sb, int64_t sn, int64_t sh,
                int box_rows = TILE) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh), static_cast<cuuint64_t>(sn), static_cast<cuuint64_t>(sb)};
  cuuint32_t box[4] = {128, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ALIGN;
}

// Paged cache [num_pages, page_size, H, d] viewed as (channel, row, head, page)
// for the head-group decode: boxes of 64 channels x 16 rows x 8 heads, which land
// in shared memory as 128 rows of 128 bytes, head-major (16 rows per head).
int make_map_heads(CUtensorMap* m, const void* ptr, int pages, int page_size, int H, int d, int64_t sb, int64_t sn,
                   int64_t sh, int box_rows, int box_heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn) * 2, static_cast<cuuint64_t>(sh) * 2,
                           static_cast<cuuint64_t>(sb) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_heads), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ALIGN;
}

// ---- argument checks ----------------------------------------------------------------
int check_shape(const fa_shape_t* s) {
  if (!s) return FA_ERR_INVALID;
  if (s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->Nq <= 0 || s->Nk <= 0) return FA_ERR_INVALID;
  if (s->Hq % s->Hkv != 0) return FA_ERR_INVALID;
  if (s->d != 64 && s->d != 128) return FA_ERR_INVALID;
  if (!(s->scale > 0.f) || !isfinite(s->scale)) return FA_ERR_INVALID;
  if (s->causal != 0 && s->causal != 1) return FA_ERR_INVALID;
  if (s->causal && s->Nq != s->Nk) return FA_ERR_INVALID;
  if (s->window != 0 && s->window != 1) return FA_ERR_INVALID;
  if (s->window && s->Nq != s->Nk) return FA_ERR_INVALID;
  if (!(s->rescale_threshold >= 0.f && s->rescale_threshold <= 16.f)) return FA_ERR_INVALID;
  // index arithmetic inside the kernels is 32-bit per (head, row) and 64-bit per element
  if (static_cast<int64_t>(s->B) * s->Hq * s->Nq > (1ll << 31) - 1) return FA_ERR_INVALID;
  if (static_cast<int64_t>(s->Nk) > (1ll << 30)) return FA_ERR_INVALID;
  return FA_OK;
}

int check_tensor(const fa_tensor_t* t) {
  if (!t || !t->ptr) return FA_ERR_INVALID;
  if (t->stride_b < 0 || t->stride_n < 0 || t->stride_h < 0) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(t->ptr) & 15) != 0) return FA_ERR_ALIGN;
  if ((t->stride_b % 8) || (t->stride_n % 8) || (t->stride_h % 8)) return FA_ERR_ALIGN;
  return FA_OK;
}

// one-byte E4M3 codes: TMA and the quantiser's 16-byte row accesses need 16-byte strides
int check_tensor_u8(const fa_tensor_t* t) {
  if (!t || !t->ptr) return FA_ERR_INVALID;
  if (t->stride_b < 0 || t->stride_n < 0 || t->stride_h < 0) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(t->ptr) & 15) != 0) return FA_ERR_ALIGN;
  if ((t->stride_b % 16) || (t->stride_n % 16) || (t->stride_h % 16)) return FA_ERR_ALIGN;
  return FA_OK;
}

int check_ws(const void* ws, size_t have, size_t need) {
  if (!ws || have < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 15) != 0) return FA_ERR_ALIGN;
  return FA_OK;
}

Dims dims_of(const fa_shape_t* s) {
  int wl = UNBOUNDED, wr = UNBOUNDED;
  if (s->window) {
    if (s->window_left >= 0) wl = imin(s->window_left, UNBOUNDED);
    if (s->window_right >= 0) wr = imin(s->window_right, UNBOUNDED);
  }
  if (s->causal) wr = imin(wr, 0);
  return Dims{s->B, s->Hq, s->Hkv, s->Nq, s->Nk, s->causal, wl, wr};
}

OutRows rows_of(const fa_tensor_t* t) { return OutRows{t->ptr, t->stride_b, t->stride_n, t->stride_h}; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every call starts by clearing the workspace header (status word and unit
// counters), so the status read later belongs to the most recent call.
int clear_header(void* ws, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws, 0, FA_WS_HEADER_BYTES, st);
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_CUDA);
}

int nq_pad(const fa_shape_t* s) { return cdiv(s->Nq, TILE) * TILE; }

// decode: resolve the requested split count (0 = auto) to the number used
int decode_splits_resolved(const fa_shape_t* s, int requested, int sms) {
  const int tiles = cdiv(s->Nk, TILE);
  int S = requested;
  if (S <= 0) {
    // one CTA per SM at a time: minimise (waves x (tiles per split + pipeline
    // ramp of ~2 tiles)), with a small charge per split for the combine
    const int units = s->B * s->Hkv;
    int best = 1;
    double best_cost = 1e30;
    for (int c = 1; c <= 256 && c <= tiles; ++c) {
      const int ctas = units * c;
      const int waves = cdiv(ctas, sms > 0 ? sms : 1);
      const double cost = static_cast<double>(waves) * (cdiv(tiles, c) + 2) + 0.01 * c;
      if (cost < best_cost) {
        best_cost = cost;
        best = c;
      }
    }
    S = best;
  }
  if (S > tiles) S = tiles;
  return decode_nsplits(s->Nk, S);
}

// The head-group paged decode: K/V heads per CTA (0: the per-head kernel).  Eight
// when Hkv is a multiple of 8 and pages are whole 16-row slices; four or two when
// pages hold 16, 32 or 64 rows (with pages of whole tiles the per-head kernel's
// boxes are already 16 KB).  One 16-row tile of packed rows per head.
int decode_head_group(const fa_shape_t* s, int page_size) {
  if ((s->Hq / s->Hkv) * s->Nq > 16 || page_size % 16 != 0) return 0;
  if (s->Hkv % DECODE_HEAD_GROUP == 0) return DECODE_HEAD_GROUP;
  if (page_size >= TILE) return 0;
  return s->Hkv % 4 == 0 ? 4 : s->Hkv % 2 == 0 ? 2 : 0;
}

// Its splits per sequence: the same cost model over stages of 128 / hg keys, with
// B * Hkv / hg CTAs per split.
int decode_splits_hg(const fa_shape_t* s, int requested, int sms, int hg) {
  const int slices = cdiv(s->Nk, TILE / hg);
  int S = requested;
  if (S <= 0) {
    const int units = s->B * (s->Hkv / hg);
    int best = 1;
    double best_cost = 1e30;
    for (int c = 1; c <= 1024 && c <= slices; ++c) {
      const int waves = cdiv(units * c, sms > 0 ? sms : 1);
      const double cost = static_cast<double>(waves) * (cdiv(slices, c) + 4) + 0.02 * c;
      if (cost < best_cost) {
        best_cost = cost;
        best = c;
      }
    }
    S = best;
  }
  return S > slices ? slices : S;
}

size_t decode_ws_bytes(const fa_shape_t* s, int S) {
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * s->Nq * S;
  return FA_WS_HEADER_BYTES + round_up(rows * sizeof(float), 256) + round_up(rows * s->d * sizeof(float), 256);
}

}  // namespace

extern "C" {

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument (null pointer, size, Hq % Hkv, head dim, causal with Nq != Nk)";
    case FA_ERR_ALIGN: return "misaligned tensor (pointer must be 16-byte aligned, strides multiples of 8 elements)";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_ARCH: return "current CUDA device is not an sm_103 (GB300) GPU";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case FA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case FA_ERR_TOO_LARGE: return "problem needs more scratch than the fixed no-allocation array holds";
    default: return "unknown error";
  }
}

int fa_last_cuda_error(void) { return g_last_cuda_error; }

void fa_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns > 0 ? ns : 1; }

void fa_test_withhold_arrive(void) { g_withhold = true; }

void fa_set_trace(void* buf, size_t bytes) {
  g_trace = bytes > 0 ? buf : nullptr;
  g_trace_bytes = buf ? bytes : 0;
}

// ------------------------------------------------------------------------ plans
int fa_tile_class(const fa_shape_t* s, int qt, int kt) {
  if (check_shape(s) != FA_OK) return -1;
  const Dims d = dims_of(s);
  if (qt < 0 || kt < 0 || qt >= q_tiles(d) || kt >= k_tiles(d)) return -1;
  return tile_class(d, qt, kt);
}

int fa_fwd_num_units(const fa_shape_t* s) { return check_shape(s) == FA_OK ? fwd_units(dims_of(s)) : -1; }
int fa_dkdv_num_units(const fa_shape_t* s) { return check_shape(s) == FA_OK ? dkdv_units(dims_of(s)) : -1; }
int fa_dq_num_units(const fa_shape_t* s) { return check_shape(s) == FA_OK ? dq_units(dims_of(s)) : -1; }

int fa_fwd_unit(const fa_shape_t* s, int i, int* b, int* h, int* p) {
  if (check_shape(s) != FA_OK || !b || !h || !p) return FA_ERR_INVALID;
  const Dims d = dims_of(s);
  if (i < 0 || i >= fwd_units(d)) return FA_ERR_INVALID;
  fwd_unit(d, i, *b, *h, *p);
  return FA_OK;
}

int fa_dkdv_unit(const fa_shape_t* s, int i, int* b, int* kvh, int* kt) {
  if (check_shape(s) != FA_OK || !b || !kvh || !kt) return FA_ERR_INVALID;
  const Dims d = dims_of(s);
  if (i < 0 || i >= dkdv_units(d)) return FA_ERR_INVALID;
  dkdv_unit(d, i, *b, *kvh, *kt);
  return FA_OK;
}

int fa_dq_unit(const fa_shape_t* s, int i, int* b, int* h, int* qt) {
  if (check_shape(s) != FA_OK || !b || !h || !qt) return FA_ERR_INVALID;
  const Dims d = dims_of(s);
  if (i < 0 || i >= dq_units(d)) return FA_ERR_INVALID;
  dq_unit(d, i, *b, *h, *qt);
  return FA_OK;
}

int fa_fwd_schedule(const fa_shape_t* s, int grid, int* start, int* ord) {
  if (check_shape(s) != FA_OK || !start || !ord) return FA_ERR_INVALID;
  const FwdSched* sc = causal_schedule(dims_of(s), s->d, false, grid);
  if (!sc) return FA_ERR_INVALID;
  for (int c = 0; c <= grid; ++c) start[c] = sc->start[c];
  for (int k = 0; k < sc->start[grid]; ++k) ord[k] = sc->ord[k];
  return FA_OK;
}

int fa_fwd_split_plan(const fa_shape_t* s, int sms, int* split0, int* nsplit) {
  if (check_shape(s) != FA_OK || sms < 1 || !split0 || !nsplit) return FA_ERR_INVALID;
  const Dims d = dims_of(s);
  if (mask_kind(d) != MASK_NONE) return FA_ERR_INVALID;
  const FwdSplit sp = fwd_split_plan(d, sms);
  *split0 = sp.split0;
  *nsplit = sp.nsplit;
  return FA_OK;
}

int fa_decode_split_range(const fa_shape_t* s, int num_splits, int i, int* start, int* end) {
  if (check_shape(s) != FA_OK || num_splits <= 0 || !start || !end) return FA_ERR_INVALID;
  const int n = decode_nsplits(s->Nk, num_splits);
  if (i < 0 || i >= n) return FA_ERR_INVALID;
  const int chunk = decode_chunk(s->Nk, num_splits);
  *start = i * chunk;
  *end = imin(s->Nk, (i + 1) * chunk);
  return FA_OK;
}

// ------------------------------------------------------------------------ status
int fa_get_device_status(void* ws, void* stream, int* status) {
  if (!ws || !status) return FA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_CUDA);
  int v = 0;
  e = cudaMemcpy(&v, static_cast<char*>(ws) + FA_WS_STATUS_OFFSET, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_CUDA);
  e = cudaMemset(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_CUDA);
  *status = v;
  if (v & FA_STATUS_TIMEOUT_MASK) return FA_ERR_TIMEOUT;
  return (v & FA_STATUS_BAD_INPUT) ? FA_ERR_INVALID : FA_OK;
}

// ------------------------------------------------------------------------ forward
// Bytes of key-split partials an unmasked dense forward needs on this device (0:
// it runs no split units), and the plan they come from.
size_t fwd_split_bytes(const fa_shape_t* s, FwdSplit* plan) {
  const Dims dm = dims_of(s);
  if (mask_kind(dm) != MASK_NONE) return 0;
  int sms = 0;
  if (device_info(&sms) != FA_OK) return 0;
  const FwdSplit sp = fwd_split_plan(dm, sms);
  if (sp.nsplit < 2) return 0;
  if (plan) *plan = sp;
  const size_t rows = static_cast<size_t>(fwd_units(dm) - sp.split0) * sp.nsplit * 2 * TILE;
  return round_up(rows * sizeof(float), 256) + rows * s->d * sizeof(float);
}

size_t fa_fwd_workspace_size(const fa_shape_t* s) {
  return check_shape(s) == FA_OK ? FA_WS_HEADER_BYTES + fwd_split_bytes(s, nullptr) : 0;
}

// Packed variable-length sequences: the cu arrays (device) and the longest
// lengths; shape Nq / Nk are then the packed tensors' token counts.
struct Packed {
  const int* cu_q;
  const int* cu_k;
  int max_q, max_k;
};

int check_packed(const fa_shape_t* s, const Packed* pk) {
  if (!pk) return FA_OK;
  if (!pk->cu_q || !pk->cu_k || s->window) return FA_ERR_INVALID;
  if (pk->max_q < 1 || pk->max_q > s->Nq || pk->max_k < 1 || pk->max_k > s->Nk) return FA_ERR_INVALID;
  return FA_OK;
}

// Dims of the kernels: dense, or packed (the unit grid sized by the longest sequence).
Dims kernel_dims(const fa_shape_t* s, const Packed* pk) {
  Dims d = dims_of(s);
  if (pk) {
    d.Nq = pk->max_q;
    d.Nk = pk->max_k;
    d.cu_q = pk->cu_q;
    d.cu_k = pk->cu_k;
    d.total_q = s->Nq;
    d.total_k = s->Nk;
  }
  return d;
}

// TMA map over a dense [B, N, H, d] tensor, or a packed [total, H, d] one (B = 1).
int map_of(CUtensorMap* m, const fa_tensor_t* t, const fa_shape_t* s, int n, int h, const Packed* pk) {
  if (pk) return make_map(m, t->ptr, 1, n, h, s->d, static_cast<int64_t>(n) * t->stride_n, t->stride_n, t->stride_h);
  return make_map(m, t->ptr, s->B, n, h, s->d, t->stride_b, t->stride_n, t->stride_h);
}

OutRows out_rows(const fa_tensor_t* t, const Packed* pk) {
  return OutRows{t->ptr, pk ? 0 : t->stride_b, t->stride_n, t->stride_h};
}

// Block-sparse table (CSR over 128-row query tiles and 128-key tiles).
struct Sparse {
  const int* row_ptr;
  const int* col_idx;
  int nnz;
};

// Workspace of the packed forward: the header, then the device-side work plan.
size_t fwd_varlen_ws_bytes(const fa_shape_t* s, int max_q) {
  const int levels = cdiv(cdiv(max_q, TILE), 2);
  return FA_WS_HEADER_BYTES + round_up(static_cast<size_t>(varlen_plan_ints(levels, s->B)) * sizeof(int), 256);
}

int fwd_impl(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o, float* lse,
             const fa_tensor_t* o_res, const fa_shape_t* s, const Packed* pk, void* ws, size_t ws_bytes,
             void* stream, const Sparse* sp = nullptr) {
  int rc;
  if ((rc = check_shape(s)) || (rc = check_packed(s, pk)) || (rc = check_tensor(q)) || (rc = check_tensor(k)) ||
      (rc = check_tensor(v)) || (rc = check_tensor(o)) || (o_res && (rc = check_tensor(o_res))))
    return rc;
  if (!lse) return FA_ERR_INVALID;
  if ((rc = check_ws(ws, ws_bytes, pk ? fwd_varlen_ws_bytes(s, pk->max_q) : fa_fwd_workspace_size(s)))) return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  FwdLaunch a;
  memset(&a, 0, sizeof(a));
  a.dims = kernel_dims(s, pk);
  a.d = s->d;
  a.scale = s->scale;
  a.tau = s->rescale_threshold;
  if ((rc = map_of(&a.tm_q, q, s, s->Nq, s->Hq, pk)) || (rc = map_of(&a.tm_k, k, s, s->Nk, s->Hkv, pk)) ||
      (rc = map_of(&a.tm_v, v, s, s->Nk, s->Hkv, pk)))
    return rc;
  a.o = out_rows(o, pk);
  a.o_res = o_res ? out_rows(o_res, pk) : OutRows{nullptr, 0, 0, 0};
  if (!pk && !sp) {  // dense: the outputs leave through TMA stores
    if ((rc = make_store_map(&a.tm_o, o->ptr, s->B, s->Nq, s->Hq, s->d, o->stride_b, o->stride_n, o->stride_h)))
      return rc;
    if (o_res && (rc = make_store_map(&a.tm_r, o_res->ptr, s->B, s->Nq, s->Hq, s->d, o_res->stride_b,
                                      o_res->stride_n, o_res->stride_h)))
      return rc;
    a.tma_out = 1;
  }
  if (sp) {
    a.row_ptr = sp->row_ptr;
    a.col_idx = sp->col_idx;
    a.nnz = sp->nnz;
  }
  if (pk) a.plan = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_HEADER_BYTES);
  if (!pk && !sp) a.sched = causal_schedule(a.dims, s->d, false, imax(1, imin(fwd_units(a.dims), sms)));
  FwdSplit split{0, 1};
  if (!pk && !sp && fwd_split_bytes(s, &split) > 0) {  // the last wave's units run as key-split parts
    const size_t rows = static_cast<size_t>(fwd_units(a.dims) - split.split0) * split.nsplit * 2 * TILE;
    char* base = static_cast<char*>(ws) + FA_WS_HEADER_BYTES;
    a.split0 = split.split0;
    a.nsplit = split.nsplit;
    a.part_lse = reinterpret_cast<float*>(base);
    a.part_o = reinterpret_cast<float*>(base + round_up(rows * sizeof(float), 256));
  }
  if (g_trace && !pk && !sp && s->d == 128 && sms <= TRACE_MAX_CTAS &&
      g_trace_bytes >= sizeof(unsigned long long) *
                           (TRACE_UNIT0 + static_cast<size_t>(fwd_units(a.dims)) * TRACE_UNIT_WORDS)) {
    a.trace = static_cast<unsigned long long*>(g_trace);
    a.diag = DG_TRACE;
  }
  if (g_withhold && !pk && !sp && s->d == 128 && !s->window) {
    a.diag = DG_WITHHOLD;
    g_withhold = false;
  }
  a.lse = lse;
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  a.counter = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_COUNTER_OFFSET);
  a.timeout_ns = g_timeout_ns;
  a.num_sms = sms;
  cudaError_t e = launch_header_clear(ws, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_LAUNCH);
  e = launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

int fa_fwd(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o, float* lse,
           const fa_tensor_t* o_res, const fa_shape_t* s, void* ws, size_t ws_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, o_res, s, nullptr, ws, ws_bytes, stream);
}

size_t fa_fwd_varlen_workspace_size(const fa_shape_t* s, int max_seqlen_q) {
  if (check_shape(s) != FA_OK || max_seqlen_q < 1 || max_seqlen_q > s->Nq) return 0;
  return fwd_varlen_ws_bytes(s, max_seqlen_q);
}

int fa_fwd_blocksparse(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* row_ptr,
                       const int* col_idx, int nnz, const fa_tensor_t* o, float* lse, const fa_tensor_t* o_res,
                       const fa_shape_t* s, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_shape(s))) return rc;
  if (!row_ptr || nnz < 0 || (nnz > 0 && !col_idx) || s->window || cdiv(s->Nk, TILE) > 1024) return FA_ERR_INVALID;
  const Sparse sp{row_ptr, col_idx, nnz};
  return fwd_impl(q, k, v, o, lse, o_res, s, nullptr, ws, ws_bytes, stream, &sp);
}

int fa_fwd_varlen(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, const fa_tensor_t* o, float* lse,
                  const fa_tensor_t* o_res, const fa_shape_t* s, void* ws, size_t ws_bytes, void* stream) {
  const Packed pk{cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k};
  return fwd_impl(q, k, v, o, lse, o_res, s, &pk, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------ FP8
size_t fa_quantize_fp8_workspace_size(int B, int H) {
  if (B <= 0 || H <= 0) return 0;
  return FA_WS_HEADER_BYTES + round_up(static_cast<size_t>(B) * H * sizeof(unsigned), 256);
}

int fa_quantize_fp8(const fa_tensor_t* x, int B, int N, int H, int d, int block_rows, const float* signs,
                    const fa_tensor_t* out, float* scales, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if (B <= 0 || N <= 0 || H <= 0 || (d != 64 && d != 128) || (block_rows != 0 && block_rows != TILE) || !scales)
    return FA_ERR_INVALID;
  if (static_cast<int64_t>(cdiv(N, TILE)) > 0x7fffffff || H > 65535 || B > 65535) return FA_ERR_INVALID;
  if ((rc = check_tensor(x)) || (rc = check_tensor_u8(out))) return rc;
  if ((rc = check_ws(ws, ws_bytes, fa_quantize_fp8_workspace_size(B, H)))) return rc;
  QuantLaunch a;
  memset(&a, 0, sizeof(a));
  a.x = x->ptr;
  a.sb = x->stride_b;
  a.sn = x->stride_n;
  a.sh = x->stride_h;
  a.B = B;
  a.N = N;
  a.H = H;
  a.d = d;
  a.signs = signs;
  a.out = out->ptr;
  a.ob = out->stride_b;
  a.on = out->stride_n;
  a.oh = out->stride_h;
  a.scales = scales;
  a.head_amax = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + FA_WS_HEADER_BYTES);
  a.nblk = cdiv(N, TILE);
  a.per_block = block_rows != 0;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  a.num_sms = sms;
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  a.timeout_ns = g_timeout_ns;
  if ((rc = make_map(&a.tm_x, x->ptr, B, N, H, d, x->stride_b, x->stride_n, x->stride_h))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = clear_header(ws, st))) return rc;
  if (!a.per_block) {
    cudaError_t e = cudaMemsetAsync(a.head_amax, 0, static_cast<size_t>(B) * H * sizeof(unsigned), st);
    if (e != cudaSuccess) return cuda_fail(e, FA_ERR_CUDA);
  }
  cudaError_t e = launch_quantize(a, st);
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

int fa_fwd_fp8(const fa_tensor_t* q8, const fa_tensor_t* k8, const fa_tensor_t* v8, const float* q_scale,
               const float* k_scale, const float* v_scale, const fa_tensor_t* o, float* lse, const fa_shape_t* s,
               void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_shape(s)) || (rc = check_tensor_u8(q8)) || (rc = check_tensor_u8(k8)) ||
      (rc = check_tensor_u8(v8)) || (rc = check_tensor(o)))
    return rc;
  if (s->d != 128 || !lse || !q_scale || !k_scale || !v_scale) return FA_ERR_INVALID;
  if ((rc = check_ws(ws, ws_bytes, fa_fwd_workspace_size(s)))) return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  FwdLaunch a;
  memset(&a, 0, sizeof(a));
  a.dims = dims_of(s);
  a.d = s->d;
  a.scale = s->scale;
  a.tau = s->rescale_threshold;
  if ((rc = make_map_u8(&a.tm_q, q8->ptr, s->B, s->Nq, s->Hq, s->d, q8->stride_b, q8->stride_n, q8->stride_h)) ||
      (rc = make_map_u8(&a.tm_k, k8->ptr, s->B, s->Nk, s->Hkv, s->d, k8->stride_b, k8->stride_n, k8->stride_h)) ||
      (rc = make_map_u8(&a.tm_v, v8->ptr, s->B, s->Nk, s->Hkv, s->d, v8->stride_b, v8->stride_n, v8->stride_h)))
    return rc;
  a.o = rows_of(o);
  a.o_res = OutRows{nullptr, 0, 0, 0};
  if ((rc = make_store_map(&a.tm_o, o->ptr, s->B, s->Nq, s->Hq, s->d, o->stride_b, o->stride_n, o->stride_h)))
    return rc;
  a.tma_out = 1;
  a.lse = lse;
  a.sq = q_scale;
  a.sk = k_scale;
  a.sv = v_scale;
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  a.counter = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_COUNTER_OFFSET);
  a.timeout_ns = g_timeout_ns;
  a.num_sms = sms;
  a.sched = causal_schedule(a.dims, s->d, true, imax(1, imin(fwd_units(a.dims), sms)));
  cudaError_t e = launch_header_clear(ws, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, FA_ERR_LAUNCH);
  e = launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

// ------------------------------------------------------------------------ backward
size_t bwd_ws_bytes(const fa_shape_t* s, int nq_rows) {
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * (cdiv(nq_rows, TILE) * TILE);
  return FA_WS_HEADER_BYTES + 2 * round_up(rows * sizeof(float), 256);
}

size_t fa_bwd_workspace_size(const fa_shape_t* s) {
  if (check_shape(s) != FA_OK) return 0;
  return bwd_ws_bytes(s, s->Nq);
}

// The packed backward adds the device-side work plans of its dQ and dK/dV
// kernels (the latter sized by the packed key count, a bound on the longest).
size_t bwd_plan_bytes(const fa_shape_t* s, int max_q) {
  return round_up(static_cast<size_t>(varlen_plan_ints(cdiv(max_q, TILE), s->B)) * sizeof(int), 256) +
         round_up(static_cast<size_t>(varlen_plan_ints(cdiv(s->Nk, TILE), s->B)) * sizeof(int), 256);
}

size_t fa_bwd_varlen_workspace_size(const fa_shape_t* s, int max_seqlen_q) {
  if (check_shape(s) != FA_OK || max_seqlen_q < 1 || max_seqlen_q > s->Nq) return 0;
  return bwd_ws_bytes(s, max_seqlen_q) + bwd_plan_bytes(s, max_seqlen_q);
}

// The block-sparse backward adds the two filtered lists, the dK/dV segment
// plan and the pool of partial tiles.  Split key tiles hold fewer than
// min(2 P, W / 16) partial tiles in all (P = SP_PLAN_PARALLELISM, W = the
// iterations of all heads, at most B * Hkv * (Hq / Hkv) * nnz; fa_sparse.cu).
size_t sparse_pool_slots(const fa_shape_t* s, int nnz) {
  const size_t w = static_cast<size_t>(s->B) * s->Hkv * (s->Hq / s->Hkv) * static_cast<size_t>(nnz);
  const size_t bound = (w + 15) / 16;
  return bound < 2 * SP_PLAN_PARALLELISM ? bound : 2 * SP_PLAN_PARALLELISM;
}

size_t bwd_sparse_bytes(const fa_shape_t* s, int nnz) {
  const size_t nqt = cdiv(s->Nq, TILE), nkt = cdiv(s->Nk, TILE);
  return round_up((nqt + 1) * sizeof(int), 256) + round_up((nkt + 1) * sizeof(int), 256) +
         2 * round_up(static_cast<size_t>(nnz) * sizeof(int) + 4, 256) +
         round_up(SP_PLAN_INTS * sizeof(int), 256) +
         sparse_pool_slots(s, nnz) * TILE * 2 * s->d * sizeof(float);
}

static int bwd_impl(int parts, const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v,
                    const fa_tensor_t* o, const float* lse, const fa_tensor_t* o_res, const fa_tensor_t* dout,
                    const fa_tensor_t* dq, const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* s,
                    const Packed* pk, void* ws, size_t ws_bytes, void* stream, const Sparse* sp = nullptr) {
  int rc;
  if ((rc = check_shape(s)) || (rc = check_packed(s, pk)) || (rc = check_tensor(q)) || (rc = check_tensor(k)) ||
      (rc = check_tensor(v)) ||
      (rc = check_tensor(o)) || (rc = check_tensor(dout)) || (rc = check_tensor(dq)) || (rc = check_tensor(dk)) ||
      (rc = check_tensor(dv)) || (o_res && (rc = check_tensor(o_res))))
    return rc;
  if (!lse) return FA_ERR_INVALID;
  const int nq_rows = pk ? pk->max_q : s->Nq;
  if ((rc = check_ws(ws, ws_bytes,
                     bwd_ws_bytes(s, nq_rows) + (pk ? bwd_plan_bytes(s, pk->max_q) : 0) +
                         (sp ? bwd_sparse_bytes(s, sp->nnz) : 0))))
    return rc;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  BwdLaunch a;
  memset(&a, 0, sizeof(a));
  a.dims = kernel_dims(s, pk);
  a.d = s->d;
  a.scale = s->scale;
  if ((rc = map_of(&a.tm_q, q, s, s->Nq, s->Hq, pk)) || (rc = map_of(&a.tm_k, k, s, s->Nk, s->Hkv, pk)) ||
      (rc = map_of(&a.tm_v, v, s, s->Nk, s->Hkv, pk)) || (rc = map_of(&a.tm_do, dout, s, s->Nq, s->Hq, pk)))
    return rc;
  a.o = out_rows(o, pk);
  a.o_res = o_res ? out_rows(o_res, pk) : OutRows{nullptr, 0, 0, 0};
  a.dout = out_rows(dout, pk);
  a.dq = out_rows(dq, pk);
  a.dk = out_rows(dk, pk);
  a.dv = out_rows(dv, pk);
  if (!pk && !sp) {  // dense: dK and dV leave through TMA stores
    if ((rc = make_store_map(&a.tm_dk, dk->ptr, s->B, s->Nk, s->Hkv, s->d, dk->stride_b, dk->stride_n,
                             dk->stride_h)) ||
        (rc = make_store_map(&a.tm_dv, dv->ptr, s->B, s->Nk, s->Hkv, s->d, dv->stride_b, dv->stride_n,
                             dv->stride_h)))
      return rc;
    a.tma_out = 1;
  }
  a.lse = lse;
  a.nq_pad = cdiv(nq_rows, TILE) * TILE;
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * a.nq_pad;
  char* base = static_cast<char*>(ws);
  a.neg_lse2 = reinterpret_cast<float*>(base + FA_WS_HEADER_BYTES);
  a.neg_delta = reinterpret_cast<float*>(base + FA_WS_HEADER_BYTES + round_up(rows * sizeof(float), 256));
  SparseLaunch sl;
  memset(&sl, 0, sizeof(sl));
  if (sp) {  // the caller's table -> filtered per-query-tile and per-key-tile lists in the workspace
    char* w = base + bwd_ws_bytes(s, nq_rows);
    const int nqt = cdiv(s->Nq, TILE), nkt = cdiv(s->Nk, TILE);
    sl.row_ptr = sp->row_ptr;
    sl.col_idx = sp->col_idx;
    sl.nnz = sp->nnz;
    sl.nqt = nqt;
    sl.nkt = nkt;
    sl.causal = s->causal;
    sl.group = s->Hq / s->Hkv;
    sl.heads = s->B * s->Hkv;
    sl.pool_slots = static_cast<int>(sparse_pool_slots(s, sp->nnz));
    sl.rows_ptr = reinterpret_cast<int*>(w);
    w += round_up((nqt + 1) * sizeof(int), 256);
    sl.cols_ptr = reinterpret_cast<int*>(w);
    w += round_up((nkt + 1) * sizeof(int), 256);
    sl.rows_idx = reinterpret_cast<int*>(w);
    w += round_up(static_cast<size_t>(sp->nnz) * sizeof(int) + 4, 256);
    sl.cols_idx = reinterpret_cast<int*>(w);
    w += round_up(static_cast<size_t>(sp->nnz) * sizeof(int) + 4, 256);
    sl.dkdv_plan = reinterpret_cast<int*>(w);
    w += round_up(SP_PLAN_INTS * sizeof(int), 256);
    a.sp_plan = sl.dkdv_plan;
    a.sp_pool = reinterpret_cast<float*>(w);
    a.rows_ptr = sl.rows_ptr;
    a.rows_idx = sl.rows_idx;
    a.cols_ptr = sl.cols_ptr;
    a.cols_idx = sl.cols_idx;
  }
  if (pk) {
    char* plans = base + bwd_ws_bytes(s, nq_rows);
    a.plan_dq = reinterpret_cast<int*>(plans);
    a.plan_dkdv = reinterpret_cast<int*>(
        plans + round_up(static_cast<size_t>(varlen_plan_ints(cdiv(pk->max_q, TILE), s->B)) * sizeof(int), 256));
  }
  a.status = reinterpret_cast<int*>(base + FA_WS_STATUS_OFFSET);
  a.counters = reinterpret_cast<int*>(base + FA_WS_COUNTER_OFFSET);
  a.timeout_ns = g_timeout_ns;
  a.num_sms = sms;
  a.parts = parts;
  cudaError_t e = launch_header_clear(ws, static_cast<cudaStream_t>(stream));
  if (sp && e == cudaSuccess) {
    sl.status = a.status;
    e = launch_sparse_lists(sl, static_cast<cudaStream_t>(stream));
  }
  if (e == cudaSuccess) e = launch_bwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

size_t fa_bwd_blocksparse_workspace_size(const fa_shape_t* s, int nnz) {
  if (check_shape(s) != FA_OK || nnz < 0) return 0;
  return bwd_ws_bytes(s, s->Nq) + bwd_sparse_bytes(s, nnz);
}

int fa_bwd_blocksparse(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* row_ptr,
                       const int* col_idx, int nnz, const fa_tensor_t* o, const float* lse,
                       const fa_tensor_t* o_res, const fa_tensor_t* dout, const fa_tensor_t* dq,
                       const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* s, void* ws, size_t ws_bytes,
                       void* stream) {
  int rc;
  if ((rc = check_shape(s))) return rc;
  if (!row_ptr || nnz < 0 || (nnz > 0 && !col_idx) || s->window || cdiv(s->Nq, TILE) > 1024 ||
      cdiv(s->Nk, TILE) > 1024)
    return FA_ERR_INVALID;
  const Sparse sp{row_ptr, col_idx, nnz};
  return bwd_impl(7, q, k, v, o, lse, o_res, dout, dq, dk, dv, s, nullptr, ws, ws_bytes, stream, &sp);
}

int fa_bwd(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o,
           const float* lse, const fa_tensor_t* o_res, const fa_tensor_t* dout, const fa_tensor_t* dq,
           const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* s, void* ws, size_t ws_bytes,
           void* stream) {
  return bwd_impl(7, q, k, v, o, lse, o_res, dout, dq, dk, dv, s, nullptr, ws, ws_bytes, stream);
}

int fa_bwd_varlen(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, const fa_tensor_t* o,
                  const float* lse, const fa_tensor_t* o_res, const fa_tensor_t* dout, const fa_tensor_t* dq,
                  const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* s, void* ws, size_t ws_bytes,
                  void* stream) {
  const Packed pk{cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k};
  return bwd_impl(7, q, k, v, o, lse, o_res, dout, dq, dk, dv, s, &pk, ws, ws_bytes, stream);
}

int fa_bwd_part(int part, const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o,
                const float* lse, const fa_tensor_t* o_res, const fa_tensor_t* dout, const fa_tensor_t* dq,
                const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* s, void* ws, size_t ws_bytes,
                void* stream) {
  if (part < 0 || part > 2) return FA_ERR_INVALID;
  return bwd_impl(1 << part, q, k, v, o, lse, o_res, dout, dq, dk, dv, s, nullptr, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------ decode
int fa_decode_num_splits(const fa_shape_t* s, int num_splits) {
  if (check_shape(s) != FA_OK) return -1;
  int sms = 148;
  if (num_splits <= 0 && device_info(&sms) != FA_OK) sms = 148;
  return decode_splits_resolved(s, num_splits, sms);
}

int fa_decode_partials_layout(const fa_shape_t* s, int num_splits, size_t* lse_off, size_t* o_off) {
  const int S = fa_decode_num_splits(s, num_splits);
  if (S <= 0 || !lse_off || !o_off) return FA_ERR_INVALID;
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * s->Nq * S;
  *lse_off = FA_WS_HEADER_BYTES;
  *o_off = FA_WS_HEADER_BYTES + round_up(rows * sizeof(float), 256);
  return FA_OK;
}

size_t fa_decode_workspace_size(const fa_shape_t* s, int num_splits) {
  const int S = fa_decode_num_splits(s, num_splits);
  if (S <= 0) return 0;
  return decode_ws_bytes(s, S);
}

// The paged decode's split count: the head-group grid's where it applies.
static int paged_splits(const fa_shape_t* s, int num_splits, int page_size, int sms) {
  const int hg = decode_head_group(s, page_size);
  return hg ? decode_splits_hg(s, num_splits, sms, hg) : decode_splits_resolved(s, num_splits, sms);
}

size_t fa_decode_paged_workspace_size(const fa_shape_t* s, int num_splits, int page_size) {
  if (check_shape(s) != FA_OK || page_size < 1) return 0;
  int sms = 148;
  if (num_splits <= 0 && device_info(&sms) != FA_OK) sms = 148;
  const int S = paged_splits(s, num_splits, page_size, sms);
  return S > 0 ? decode_ws_bytes(s, S) : 0;
}

int fa_decode(const fa_tensor_t* q, const fa_tensor_t* kc, const fa_tensor_t* vc, const fa_tensor_t* o,
              float* lse, const fa_shape_t* s, int num_splits, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_shape(s)) || (rc = check_tensor(q)) || (rc = check_tensor(kc)) || (rc = check_tensor(vc)) ||
      (rc = check_tensor(o)))
    return rc;
  if (!lse || s->causal || s->window) return FA_ERR_INVALID;
  if ((s->Hq / s->Hkv) * s->Nq > 64) return FA_ERR_INVALID;  // packed rows: at most four 16-row tiles
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  const int S = decode_splits_resolved(s, num_splits, sms);
  if ((rc = check_ws(ws, ws_bytes, fa_decode_workspace_size(s, num_splits)))) return rc;
  DecodeLaunch a;
  memset(&a, 0, sizeof(a));
  a.dims = dims_of(s);
  a.d = s->d;
  a.scale = s->scale;
  if ((rc = make_map(&a.tm_k, kc->ptr, s->B, s->Nk, s->Hkv, s->d, kc->stride_b, kc->stride_n, kc->stride_h)) ||
      (rc = make_map(&a.tm_v, vc->ptr, s->B, s->Nk, s->Hkv, s->d, vc->stride_b, vc->stride_n, vc->stride_h)))
    return rc;
  a.q = q->ptr;
  a.q_sb = q->stride_b;
  a.q_sn = q->stride_n;
  a.q_sh = q->stride_h;
  a.o = rows_of(o);
  a.lse = lse;
  size_t lo = 0, oo = 0;
  fa_decode_partials_layout(s, num_splits, &lo, &oo);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) + lo);
  a.o_part = reinterpret_cast<float*>(static_cast<char*>(ws) + oo);
  a.num_splits = S;
  // the chunk that yields exactly S splits
  a.chunk = decode_chunk(s->Nk, S);
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  a.timeout_ns = g_timeout_ns;
  if ((rc = clear_header(ws, static_cast<cudaStream_t>(stream)))) return rc;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

int fa_decode_paged(const fa_tensor_t* q, const fa_tensor_t* kc, const fa_tensor_t* vc, const int* block_table,
                    int max_pages, const int* seqlens_k, int num_pages, int page_size, const fa_tensor_t* o,
                    float* lse, const fa_shape_t* s, int num_splits, void* ws, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_shape(s)) || (rc = check_tensor(q)) || (rc = check_tensor(kc)) || (rc = check_tensor(vc)) ||
      (rc = check_tensor(o)))
    return rc;
  if (!lse || s->causal || s->window || !block_table || !seqlens_k || max_pages < 1 || num_pages < 1)
    return FA_ERR_INVALID;
  if ((s->Hq / s->Hkv) * s->Nq > 64) return FA_ERR_INVALID;
  // pages of 16, 32 or 64 keys stack into a 128-key tile; larger pages hold whole tiles
  const bool small = page_size == 16 || page_size == 32 || page_size == 64;
  if (!small && (page_size < TILE || page_size % TILE != 0)) return FA_ERR_INVALID;
  if (static_cast<int64_t>(max_pages) * page_size < s->Nk) return FA_ERR_INVALID;
  int sms = 0;
  if ((rc = device_info(&sms))) return rc;
  const int S = paged_splits(s, num_splits, page_size, sms);
  if ((rc = check_ws(ws, ws_bytes, decode_ws_bytes(s, S)))) return rc;
  DecodeLaunch a;
  memset(&a, 0, sizeof(a));
  a.dims = dims_of(s);
  a.d = s->d;
  a.scale = s->scale;
  a.head_group = decode_head_group(s, page_size);
  if (a.head_group) {
    const int rb = imin(page_size, TILE / a.head_group);  // box rows: a stage's keys, or a whole page
    if ((rc = make_map_heads(&a.tm_k, kc->ptr, num_pages, page_size, s->Hkv, s->d, kc->stride_b, kc->stride_n,
                             kc->stride_h, rb, a.head_group)) ||
        (rc = make_map_heads(&a.tm_v, vc->ptr, num_pages, page_size, s->Hkv, s->d, vc->stride_b, vc->stride_n,
                             vc->stride_h, rb, a.head_group)))
      return rc;
  } else {
    const int box_rows = small ? page_size : TILE;
    if ((rc = make_map(&a.tm_k, kc->ptr, num_pages, page_size, s->Hkv, s->d, kc->stride_b, kc->stride_n,
                       kc->stride_h, box_rows)) ||
        (rc = make_map(&a.tm_v, vc->ptr, num_pages, page_size, s->Hkv, s->d, vc->stride_b, vc->stride_n,
                       vc->stride_h, box_rows)))
      return rc;
  }
  a.q = q->ptr;
  a.q_sb = q->stride_b;
  a.q_sn = q->stride_n;
  a.q_sh = q->stride_h;
  a.o = rows_of(o);
  a.lse = lse;
  const size_t prow = static_cast<size_t>(s->B) * s->Hq * s->Nq * S;  // partials: [B, Hq, Nq, S]
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) + FA_WS_HEADER_BYTES);
  a.o_part = reinterpret_cast<float*>(static_cast<char*>(ws) + FA_WS_HEADER_BYTES + round_up(prow * sizeof(float), 256));
  a.num_splits = S;
  a.chunk = 0;  // per sequence, in the kernel
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  a.timeout_ns = g_timeout_ns;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seqlens = seqlens_k;
  a.num_pages = num_pages;
  a.page_size = page_size;
  if ((rc = clear_header(ws, static_cast<cudaStream_t>(stream)))) return rc;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

// ------------------------------------------------------------------------ self-test
int fa_selftest_mma(int mode, int nk, const void* a, const void* b, float* c, void* ws, void* stream) {
  if (mode < 0 || mode > 3 || (nk != 64 && nk != 128) || (mode >= 2 && nk != 128) || !a || !b || !c)
    return FA_ERR_INVALID;
  int sms = 0, rc;
  if ((rc = check_ws(ws, FA_WS_HEADER_BYTES, FA_WS_HEADER_BYTES))) return rc;
  if ((rc = device_info(&sms))) return rc;
  CUtensorMap ta, tb;
  // mode 0: a, b are [128 x k] row-major.  mode 1: a [128 x 128] is read by
  // threads (the map over it is unused), b is [128 x n] row-major.  Modes 2, 3:
  // the same with one-byte E4M3 codes.
  if (mode >= 2) {
    if ((rc = make_map_u8(&ta, mode == 2 ? a : b, 1, 128, 1, 128, 128 * 128, 128, 128)) ||
        (rc = make_map_u8(&tb, b, 1, 128, 1, 128, 128 * 128, 128, 128)))
      return rc;
  } else if ((rc = make_map(&ta, mode == 0 ? a : b, 1, 128, 1, nk, 128 * nk, nk, nk)) ||
             (rc = make_map(&tb, b, 1, 128, 1, nk, 128 * nk, nk, nk))) {
    return rc;
  }
  int* status = reinterpret_cast<int*>(static_cast<char*>(ws) + FA_WS_STATUS_OFFSET);
  if ((rc = clear_header(ws, static_cast<cudaStream_t>(stream)))) return rc;
  cudaError_t e = launch_selftest_mma(mode, nk, ta, tb, a, c, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, FA_ERR_LAUNCH);
}

}  // extern "C"
