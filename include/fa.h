/*
 * fa.h -- C ABI of libfa_gb300.so: exact IO-aware attention (FlashAttention)
 * for one GB300 GPU (sm_103a).
 *
 * The method: scaled-dot-product attention computed tile by tile with an online
 * softmax, so the Nq x Nk score matrix never reaches HBM ("第18章 FlashAttention",
 * §18.4.1-§18.4.3; "CMU 11-868 L21 FlashAttention" notes, slides 9-12); a
 * backward pass that rebuilds P on chip from the saved log-sum-exp instead of
 * storing it (§18.4.4; lecture slide 14); and split-KV decoding
 * (FlashDecoding) with a log-sum-exp weighted combine (§18.8.2; slides 57-60).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are bf16, layout [B, N, H, d] (batch, sequence, head, head dim) as
 *    in the flash_attn_func interface of §18.7.1.  Each is passed as an
 *    fa_tensor_t: a device pointer plus the batch / sequence / head strides in
 *    ELEMENTS; the head-dim stride is 1.  Pointers must be 16-byte aligned and
 *    the three strides multiples of 8 elements (16 bytes): the kernels move
 *    tiles with the Tensor Memory Accelerator, which requires both.
 *  - LSE is fp32, contiguous [B, Hq, Nq], natural log, in units of the scaled
 *    scores: LSE_i = ln sum_j exp(scale * q_i . k_j).
 *  - Grouped-query attention: Hq must be a multiple of Hkv; query head h reads
 *    K/V head h / (Hq / Hkv) (§18.2.2; consecutive grouping).
 *  - d is 64 or 128.  scale must be finite and > 0 (callers usually pass
 *    1/sqrt(d), §18.2.1).
 *  - causal != 0 masks key j for query i when j > i (§18.2.2, top-left
 *    aligned) and requires Nq == Nk.
 *  - Ownership: the caller allocates and owns every device buffer, including
 *    the workspace (size from the matching *_workspace_size call).  The library
 *    never allocates, frees or synchronises in the compute calls; work is
 *    enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *    the call returns before it finishes.
 *  - Errors: the return value is FA_OK or an FA_ERR_* code; fa_strerror()
 *    describes it.  Argument errors are detected before anything is enqueued.
 *    Errors found on the GPU (a bounded wait that ran out) are recorded in the
 *    workspace and returned by fa_get_device_status().  Each compute call
 *    first clears the workspace's 256-byte header (status word and work
 *    counters) on its stream, so the status belongs to the latest call, and
 *    calls that share one workspace must not run concurrently.
 *  - Every device buffer must live on the current CUDA device, which must be
 *    an sm_103 part (FA_ERR_ARCH otherwise).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,   /* null pointer, bad size, Hq % Hkv != 0, d not 64/128, causal with Nq != Nk */
  FA_ERR_ALIGN = 2,     /* pointer not 16-byte aligned or stride not a multiple of 8 elements */
  FA_ERR_WORKSPACE = 3, /* workspace missing or smaller than the *_workspace_size answer */
  FA_ERR_ARCH = 4,      /* current device is not sm_103 */
  FA_ERR_LAUNCH = 5,    /* a kernel launch failed (the CUDA error is in fa_last_cuda_error) */
  FA_ERR_TIMEOUT = 6,   /* a device-side bounded wait ran out (see fa_get_device_status) */
  FA_ERR_CUDA = 7,      /* another CUDA runtime/driver call failed */
  FA_ERR_TOO_LARGE = 8  /* the problem needs more scratch than fa_decode_noalloc's fixed array holds */
};

typedef struct {
  void* ptr;          /* device pointer to the element [0, 0, 0, 0] (bf16) */
  int64_t stride_b;   /* elements between consecutive batch entries */
  int64_t stride_n;   /* elements between consecutive sequence positions */
  int64_t stride_h;   /* elements between consecutive heads; head-dim stride is 1 */
} fa_tensor_t;

typedef struct {
  int B;        /* batch */
  int Hq;       /* query heads */
  int Hkv;      /* key/value heads; Hq % Hkv == 0 */
  int Nq;       /* query length */
  int Nk;       /* key/value length */
  int d;        /* head dim: 64 or 128 */
  float scale;  /* softmax scale applied to q.k (e.g. 1/sqrt(d)) */
  int causal;   /* 0 or 1 */
  /* Sliding window (flash_attn_func's window_size, §18.7.1; local attention,
   * §18.8.1): with window = 1, query i sees keys i - window_left .. i +
   * window_right (a negative bound is unbounded; causal still caps at i).
   * window = 0 (a zero-initialised struct) means no window.  Needs Nq == Nk,
   * like causal; forward and backward only (decode rejects it). */
  int window;
  int window_left;
  int window_right;
  /* Conditional rescaling (lecture notes, FA4: a variant of the online softmax
   * that skips most rescalings of O).  The forward exponentiates each key tile
   * against a reference max that moves only when the tile's row max exceeds it
   * by more than rescale_threshold, in log2 units of the probabilities (P then
   * reaches at most 2^rescale_threshold before normalisation); O and l keep
   * their scale while it stays, so most O rescalings are skipped.  O / l and the
   * LSE stay exact up to rounding; what changes is the rounding of P: the
   * dominant P of a nearly one-hot row is no longer exactly 1.0, which costs
   * the backward accuracy there (D = dO . O from a forward O that carries that
   * rounding).  0 (a zero-initialised struct) = the exact running max; range
   * [0, 16]; FA4 uses 8.  Read by the forward calls (fa_fwd, fa_fwd_varlen,
   * fa_fwd_blocksparse, fa_fwd_fp8); the backward and decode calls ignore it. */
  float rescale_threshold;
} fa_shape_t;

/* ---------------------------------------------------------------------------
 * Forward.  "第18章" §18.4.1 (tiling: Q tiles outer, K/V tiles inner, running
 * max m and sum l), §18.4.2 (online update), §18.4.3 (kernel: O rescaled, final
 * O / l, m and l saved); Fig. 18-6 (the saved statistic is the log-sum-exp);
 * §18.5.2 (causal: key tiles above the diagonal skipped, the diagonal tile
 * masked element by element); lecture slides 26-46 (persistent kernel,
 * longest-first order of causal work).
 *   q   [B, Nq, Hq, d]  in
 *   k,v [B, Nk, Hkv, d] in
 *   o   [B, Nq, Hq, d]  out (bf16, round to nearest even)
 *   lse [B, Hq, Nq]     out (fp32, contiguous)
 *   o_residual [B, Nq, Hq, d]  optional out (NULL = not written): the bf16
 *       rounding residual of O, i.e. bf16(O_fp32 - O).  O + o_residual carries
 *       about 16 significant bits; fa_bwd uses it for D (see there).
 * Needs fa_fwd_workspace_size(shape) bytes of workspace (16-byte aligned); for
 * a shape without a mask (not causal, no window) the size depends on the
 * current device's SM count, so size the workspace on the device that runs the
 * call.  Enqueues two kernels: one that clears the workspace header, then the
 * forward, launched with programmatic stream serialisation so that its CTAs set
 * up shared memory and TMEM while the first still runs (they touch global
 * memory only after it has finished).  The forward calls below do the same.
 * Without a mask, when the work units do not fill the last wave of SMs (or
 * there are fewer units than SMs), the units of that wave run as 2-4 parts
 * along the keys (flash-decoding's split, here for a prefill), each writing its
 * normalised O and LSE to the workspace, and a third kernel merges the parts
 * by their LSE into O, the residual and LSE.  Results are bitwise the same on
 * every call for one shape on one device; on a device with another SM count
 * an unmasked shape may split differently (fa_fwd_split_plan), which changes
 * the rounding of O and LSE but not their error bound.
 * ------------------------------------------------------------------------- */
size_t fa_fwd_workspace_size(const fa_shape_t* shape);
int fa_fwd(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o, float* lse,
           const fa_tensor_t* o_residual, const fa_shape_t* shape, void* workspace, size_t workspace_bytes,
           void* stream);

/* ---------------------------------------------------------------------------
 * Block-sparse forward ("第18章" §18.8.1): a CSR table over 128-row query tiles
 * lists the 128-key tiles each one attends to; the kernel loads and computes
 * only those (the inner loop runs over the list).  row_ptr: device int32
 * [ceil(Nq/128) + 1], from 0, non-decreasing, ending at nnz; col_idx: device
 * int32 [nnz], strictly increasing within each row, each below ceil(Nk/128).
 * Key j is visible to query i iff j's tile is listed for i's tile (and, causal,
 * j <= i).  Rows that see no key get O = 0 (and a zero residual) and LSE =
 * -inf.  One table serves every batch entry and head.  Entries that break the
 * rules are skipped and reported through the workspace status
 * (fa_get_device_status -> FA_ERR_INVALID).  Nk <= 131072; no window; other
 * arguments and the workspace as fa_fwd.
 * ------------------------------------------------------------------------- */
int fa_fwd_blocksparse(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* row_ptr,
                       const int* col_idx, int nnz, const fa_tensor_t* o, float* lse,
                       const fa_tensor_t* o_residual, const fa_shape_t* shape, void* workspace,
                       size_t workspace_bytes, void* stream);
/* Block-sparse backward: dQ, dK, dV of fa_fwd_blocksparse (same table; o, lse
 * and o_residual from it).  The call first turns the table into per-query-tile
 * and per-key-tile lists in the workspace (checked as above, ascending, so the
 * results are deterministic); the dQ kernel visits each query tile's listed key
 * tiles, the dK/dV kernel each key tile's listing query tiles.  Rows that see
 * no key get dQ = 0; keys no query sees get dK = dV = 0.  Nq, Nk <= 131072.
 * A key tile listed by many query tiles (a global column) is cut into
 * segments so that no SM carries much more than its share: its g x (listing
 * query tiles) iterations are split when they exceed
 * max(32, ceil(all heads' iterations / 152)), each segment writes an fp32
 * partial tile into the workspace, and a reduce kernel sums them in segment
 * order (the split depends on the table and the shape only, so results stay
 * deterministic; unsplit tiles are written directly, as by the dense kernel).
 * Needs fa_bwd_blocksparse_workspace_size(shape, nnz) bytes (lists, the
 * segment plan and at most min(304, ceil(B Hkv (Hq/Hkv) nnz / 16)) partial
 * tiles of 128 x 2d floats). */
size_t fa_bwd_blocksparse_workspace_size(const fa_shape_t* shape, int nnz);
int fa_bwd_blocksparse(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* row_ptr,
                       const int* col_idx, int nnz, const fa_tensor_t* o, const float* lse,
                       const fa_tensor_t* o_residual, const fa_tensor_t* dout, const fa_tensor_t* dq,
                       const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* shape, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Packed variable-length sequences ("第18章" §18.7.1, flash_attn_varlen_func):
 * the B sequences of a batch lie one after another along the token axis,
 * q [total_q, Hq, d], k, v [total_k, Hkv, d] (the fa_tensor_t's stride_b is
 * ignored); sequence b is rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q
 * (cu_seqlens_k likewise of k, v), and attends only within itself, causal
 * with its own positions.  cu_seqlens_q / _k: device int32 [B + 1], starting
 * at 0, non-decreasing, ending at most at total; max_seqlen_q / _k: host ints,
 * at least every sequence's length (they size the kernels' work grid).  The
 * shape's B is the number of sequences and Nq, Nk the packed token counts
 * total_q, total_k; windows are not supported.  lse [Hq, total_q].  o,
 * o_residual, dout, dq: [total_q, Hq, d]; dk, dv: [total_k, Hkv, d].
 * Lengths the arrays cannot hold (out of range, decreasing, above max_seqlen,
 * queries with no keys, or unequal lengths under causal) are reported through
 * the workspace status (fa_get_device_status -> FA_ERR_INVALID) and those
 * sequences' outputs are not written; keys of a sequence with no queries get
 * zero gradients.  Workspaces: fa_fwd_varlen_workspace_size(shape,
 * max_seqlen_q) and fa_bwd_varlen_workspace_size(shape, max_seqlen_q); they
 * hold a work plan the call builds on the device (the units with work,
 * longest first), so no host copy of the lengths is needed.
 * ------------------------------------------------------------------------- */
size_t fa_fwd_varlen_workspace_size(const fa_shape_t* shape, int max_seqlen_q);
int fa_fwd_varlen(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, const fa_tensor_t* o, float* lse,
                  const fa_tensor_t* o_residual, const fa_shape_t* shape, void* workspace, size_t workspace_bytes,
                  void* stream);
size_t fa_bwd_varlen_workspace_size(const fa_shape_t* shape, int max_seqlen_q);
int fa_bwd_varlen(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, const fa_tensor_t* o,
                  const float* lse, const fa_tensor_t* o_residual, const fa_tensor_t* dout, const fa_tensor_t* dq,
                  const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* shape, void* workspace,
                  size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 forward ("第18章" §18.6.2; lecture notes slide 24).
 *
 * fa_quantize_fp8: E4M3 codes of a bf16 tensor x [B, N, H, d] (d = 64 or 128),
 * X_fp8 = E4M3(X / s), s = max|X| / 448 (round to nearest even, saturating
 * at 448).  block_rows = 128: one scale per 128 rows of one head (the load
 * block of the forward; use for Q and K), scales [B, H, ceil(N/128)] fp32;
 * block_rows = 0: one scale per (batch, head), scales [B, H] (use for V).
 * signs: NULL, or d device floats (+1 / -1): the rows are first rotated by
 * J = diag(signs) H_d / sqrt(d) (H_d the Sylvester Hadamard matrix), which
 * leaves Q K^T unchanged when Q and K get the same signs and spreads outlier
 * channels; the scale then includes 1 / sqrt(d).  Codes come from the
 * unnormalised transform y: inv = 448 / max|y|, code = E4M3(y * inv), each an
 * IEEE round-to-nearest fp32 operation; an all-zero block gets scale 0.
 *   out [B, N, H, d] uint8 out (strides multiples of 16 bytes)
 * Needs fa_quantize_fp8_workspace_size(B, H) bytes of workspace.
 *
 * fa_fwd_fp8: the forward of fa_fwd on E4M3 operands (d = 128 only): q8, k8
 * and v8 [.., d] uint8 codes from fa_quantize_fp8 (Q and K per block with the
 * same signs or none, V per head, unrotated), q_scale [B, Hq, ceil(Nq/128)],
 * k_scale [B, Hkv, ceil(Nk/128)], v_scale [B, Hkv] (device fp32).  S = Q K^T
 * on E4M3 tensor-core products with fp32 accumulation, times s_q s_k and the
 * shape's scale; softmax in fp32; P enters P V as E4M3(448 P) (P <= 1 fixes
 * its scale at 1/448); O = (sum E4M3(448 P) V_codes) * s_v / l -> bf16; lse as
 * in fa_fwd.  Causal and sliding windows as in fa_fwd.  Workspace as fa_fwd.
 * ------------------------------------------------------------------------- */
size_t fa_quantize_fp8_workspace_size(int B, int H);
int fa_quantize_fp8(const fa_tensor_t* x, int B, int N, int H, int d, int block_rows, const float* signs,
                    const fa_tensor_t* out, float* scales, void* workspace, size_t workspace_bytes, void* stream);
int fa_fwd_fp8(const fa_tensor_t* q8, const fa_tensor_t* k8, const fa_tensor_t* v8, const float* q_scale,
               const float* k_scale, const float* v_scale, const fa_tensor_t* o, float* lse, const fa_shape_t* shape,
               void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Backward.  §18.4.4: P rebuilt per tile from the saved statistics with no
 * rescaling, dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
 * dK = scale dS^T Q; Fig. 18-17 (dependency chain).  D_i is the full-row
 * rowsum(P o dP), which equals dO_i . O_i and is computed once before the
 * tile loops (the per-block D of the printed pseudocode is not used).  dK/dV
 * of a shared K/V head sum the contributions of its query heads.  Three
 * kernels, no atomics: preprocess (D), dK/dV (one key tile per work unit),
 * dQ (one query tile per work unit); results are deterministic.  On the dense
 * path they follow a header-clearing kernel and are launched with programmatic
 * stream serialisation: each starts while the one before it finishes and waits
 * (griddepcontrol) before it reads what that one wrote; dQ, which reads nothing
 * dK/dV writes, takes over each SM as the dK/dV kernel's CTA there finishes.
 *   q, o, dout [B, Nq, Hq, d] in;  k, v [B, Nk, Hkv, d] in;  lse in (from fa_fwd)
 *   o_residual  optional in (NULL = none): the residual written by fa_fwd.
 *       D is then dO . (O + o_residual).  Without it D is dO . O with O in
 *       bf16; when attention is nearly one-hot, dP - D is a difference of
 *       nearly equal terms and O's rounding shows up in dQ and dK (a few
 *       percent on inputs with outlier channels).
 *   dq [B, Nq, Hq, d] out;  dk, dv [B, Nk, Hkv, d] out  (bf16)
 * ------------------------------------------------------------------------- */
size_t fa_bwd_workspace_size(const fa_shape_t* shape);
int fa_bwd(const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o,
           const float* lse, const fa_tensor_t* o_residual, const fa_tensor_t* dout, const fa_tensor_t* dq,
           const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* shape, void* workspace,
           size_t workspace_bytes, void* stream);
/* The three backward launches one at a time, for callers that time or
 * schedule them separately: part 0 = preprocess (D and the padded LSE, kept in
 * the workspace), 1 = dK/dV, 2 = dQ.  Parts 1 and 2 read what part 0 left in
 * the same workspace; running parts 0, 1, 2 in order on one stream gives
 * exactly fa_bwd's results (without the overlap between its kernels).  Same
 * arguments and errors as fa_bwd; FA_ERR_INVALID for another part. */
int fa_bwd_part(int part, const fa_tensor_t* q, const fa_tensor_t* k, const fa_tensor_t* v, const fa_tensor_t* o,
                const float* lse, const fa_tensor_t* o_residual, const fa_tensor_t* dout, const fa_tensor_t* dq,
                const fa_tensor_t* dk, const fa_tensor_t* dv, const fa_shape_t* shape, void* workspace,
                size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Split-KV decode (FlashDecoding).  §18.8.2: the KV cache is cut along its
 * length into chunks processed in parallel, each producing (m_t, l_t, O_t),
 * merged by O = sum_t O_t e^{m_t-m} / sum_t l_t e^{m_t-m}; lecture slides
 * 57-60: the query heads sharing a K/V head (and the query positions) are
 * packed into the rows of matrix tiles.  Non-causal: every query row sees all
 * Nk keys.
 *   q      [B, Nq, Hq, d]   in  (Nq small: Hq/Hkv * Nq <= 64, packed into one,
 *                               two or four 16-row tiles)
 *   kcache [B, Nk, Hkv, d]  in;  vcache likewise
 *   o      [B, Nq, Hq, d]   out (bf16);  lse [B, Hq, Nq] out (fp32)
 * num_splits: requested number of KV splits, 0 = choose from the GPU's SM
 * count.  Splits are whole 128-key tiles: chunk = ceil(ceil(Nk/128)/S)*128
 * keys, split s = [s*chunk, min((s+1)*chunk, Nk)); the number used is
 * fa_decode_num_splits().  shape->causal must be 0.
 * ------------------------------------------------------------------------- */
int fa_decode_num_splits(const fa_shape_t* shape, int num_splits);
size_t fa_decode_workspace_size(const fa_shape_t* shape, int num_splits);
int fa_decode(const fa_tensor_t* q, const fa_tensor_t* kcache, const fa_tensor_t* vcache, const fa_tensor_t* o,
              float* lse, const fa_shape_t* shape, int num_splits, void* workspace, size_t workspace_bytes,
              void* stream);
/* Where fa_decode leaves the per-split partials inside its workspace (for
 * tests): lse_part [B, Hq, Nq, S] fp32 (natural log) and o_part
 * [B, Hq, Nq, S, d] fp32 (normalised by the split's own sum).  Byte offsets. */
int fa_decode_partials_layout(const fa_shape_t* shape, int num_splits, size_t* lse_offset, size_t* o_offset);

/* ---------------------------------------------------------------------------
 * Paged, variable-length decode.  §18.8.2 part 3 and §18.8.3 (PagedAttention):
 * the KV cache lives in fixed-size physical pages; logical page i of sequence
 * b is physical page block_table[b * max_pages + i], and sequence b has its own
 * length seqlens_k[b].  Sequence b's logical key r is row r % page_size of page
 * block_table[b * max_pages + r / page_size].  Otherwise as fa_decode: the same
 * q, o, lse, shape (causal 0, Hq/Hkv * Nq <= 64) and num_splits; the
 * workspace is fa_decode_paged_workspace_size(shape, num_splits, page_size)
 * bytes.
 *   kcache, vcache [num_pages, page_size, Hkv, d] bf16: stride_b = elements
 *                  between pages, stride_n between rows of a page, stride_h
 *                  between heads (16-byte aligned, multiples of 8 elements)
 *   block_table    device int32 [B, max_pages]; entries for logical pages at or
 *                  past ceil(seqlens_k[b] / page_size) are never read
 *   seqlens_k      device int32 [B], each in [1, shape->Nk]
 *   shape->Nk      the largest seqlens_k (an upper bound is fine); it sizes the
 *                  split grid; max_pages * page_size must be >= shape->Nk
 *   page_size      16, 32, 64, or a multiple of 128
 * Each sequence is cut into whole 128-key tiles by its own length, with the
 * chunk rule of fa_decode applied to seqlens_k[b]; splits past its end
 * contribute nothing.  When Hkv is a multiple of 8, page_size a multiple of
 * 16 and Hq/Hkv * Nq <= 16, one CTA serves 8 K/V heads over 16-key page slices (the copy engine
 * then moves 16 KB boxes instead of one 2 KB box per page and head): the
 * splits are whole 16-key slices, chunk = ceil(ceil(len/16)/S)*16, and S is
 * chosen for that grid when num_splits is 0.  Keys past a sequence's end are never weighted, whatever
 * the page holds there.  Device-side input errors (a length outside [1, Nk], a
 * page index outside [0, num_pages)) set a status bit that
 * fa_get_device_status() returns as FA_ERR_INVALID; such a page reads as zeros.
 * Host-side: FA_ERR_INVALID for a bad page_size, max_pages, num_pages or null
 * table/length pointers.
 * ------------------------------------------------------------------------- */
int fa_decode_paged(const fa_tensor_t* q, const fa_tensor_t* kcache, const fa_tensor_t* vcache,
                    const int* block_table, int max_pages, const int* seqlens_k, int num_pages, int page_size,
                    const fa_tensor_t* o, float* lse, const fa_shape_t* shape, int num_splits, void* workspace,
                    size_t workspace_bytes, void* stream);
/* Workspace bytes fa_decode_paged needs for (shape, num_splits, page_size); 0
 * for an invalid shape. */
size_t fa_decode_paged_workspace_size(const fa_shape_t* shape, int num_splits, int page_size);

/* ---------------------------------------------------------------------------
 * Decode without allocation.  No counterpart on the pages: this is a service
 * to callers that cannot allocate device memory, such as an inference server
 * that reserves all device memory for its own pool at start-up and forbids
 * later cudaMalloc calls (they synchronise the device and fragment the pool),
 * or a plug-in that receives only the tensors of the call.
 * fa_decode_noalloc computes exactly what fa_decode computes, with the same
 * arguments minus the workspace: its scratch (the per-split partials and the
 * status header) lives in one array of FA_DECODE_SCRATCH_BYTES compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits.  The library allocates nothing in this call.
 *  - Limit: fa_decode_workspace_size(shape, num_splits) must not exceed
 *    FA_DECODE_SCRATCH_BYTES (8 MiB; for d = 128 about
 *    B*Hq*Nq*splits*516 bytes); otherwise the call returns FA_ERR_TOO_LARGE
 *    and enqueues nothing.  Request fewer splits to fit.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents.
 *    Calls whose work overlaps on the GPU (other streams, other host threads)
 *    race on it: order them on one stream.
 *  - Errors found on the GPU (a bounded wait that ran out) are recorded in
 *    the array's header, as in a workspace: fa_decode_noalloc_status() reads
 *    and clears them (fa_get_device_status() cannot reach the array).
 * ------------------------------------------------------------------------- */
#define FA_DECODE_SCRATCH_BYTES ((size_t)8 << 20)
size_t fa_decode_noalloc_max_bytes(void);
int fa_decode_noalloc(const fa_tensor_t* q, const fa_tensor_t* kcache, const fa_tensor_t* vcache,
                      const fa_tensor_t* o, float* lse, const fa_shape_t* shape, int num_splits, void* stream);
/* Device status of the latest fa_decode_noalloc call on the current device:
 * synchronises `stream`, returns the error bits its kernels recorded in the
 * fixed array (0 = none) through *status and clears them; the return value is
 * as fa_get_device_status's (FA_ERR_TIMEOUT when a bounded wait ran out).
 * Allocates nothing. */
int fa_decode_noalloc_status(void* stream, int* status);

/* ---------------------------------------------------------------------------
 * Device status.  Synchronises `stream`, returns the error bits the kernels
 * recorded in `workspace` (0 = none) through *status, and clears them.
 * Returns FA_ERR_TIMEOUT when a bounded wait ran out, FA_ERR_INVALID when a
 * kernel found bad device-side input (paged decode), FA_OK otherwise.
 * ------------------------------------------------------------------------- */
int fa_get_device_status(void* workspace, void* stream, int* status);

/* Time budget of every device-side wait, in nanoseconds (default 10 s).  A
 * wait that runs out records an error and the kernel returns early.  */
void fa_set_wait_timeout_ns(unsigned long long ns);

/* Test hook for the bounded waits (no counterpart on the pages).  The next
 * fa_fwd call with d = 128 on dense tensors without a window runs a test
 * instantiation of the forward kernel in which one softmax warp of the CTA
 * that runs work unit 0 skips its first hand-off of P (one software mbarrier
 * arrive; no copy and no tensor-core operation is touched).  The tensor-core
 * issuer of that CTA then waits for it, and its producer for a stage the issuer
 * never frees; the first of those waits to exceed the budget
 * (fa_set_wait_timeout_ns) records its FA_STATUS_TIMEOUT_* bit, and every role
 * of the CTA leaves early: copies in flight land, TMEM is freed, and the units
 * it held are not written.
 * fa_get_device_status then returns FA_ERR_TIMEOUT.  One-shot: later calls run
 * the normal kernels.  Not thread-safe; for tests. */
void fa_test_withhold_arrive(void);

/* Diagnostics (no counterpart on the pages): timestamps of the dense forward
 * kernel, to see how its persistent CTAs spend the launch.  With a buffer set
 * (device memory, 8-byte aligned), every later fa_fwd call with d = 128 (dense
 * tensors; not the packed, block-sparse or FP8 calls) runs an instantiation of
 * the kernel that also writes %globaltimer nanoseconds into it:
 *   per CTA c < 1024:  buf[4c] start (after set-up), buf[4c+1] end (the last
 *                      of its warps to leave its role), buf[4c+2] SM id,
 *                      buf[4c+3] work units it ran;
 *   per work unit u:   buf[4096 + 16u + k], k = 0 claimed, 1 first product
 *                      issued, 2 last product issued, 3 output written, 4 CTA;
 *                      per query tile t = 0, 1 of the unit: 5 + t its first S
 *                      received, 7 + t its last P handed over, 9 + t its final
 *                      O ready, 11 + t its output written.
 * bytes must cover 8 * (4096 + 16 * units) (units: fa_fwd_num_units); otherwise
 * nothing is written.  buf = NULL or bytes = 0 turns it off.  The buffer is the
 * caller's and is overwritten by every traced call. */
void fa_set_trace(void* buf, size_t bytes);

const char* fa_strerror(int code);
/* The last CUDA runtime error code seen by the library (cudaError_t value). */
int fa_last_cuda_error(void);

/* ---------------------------------------------------------------------------
 * Host-side plans (integer, no GPU needed): exactly what the kernels use.
 * ------------------------------------------------------------------------- */
/* Causal class of query tile qt x key tile kt (128 x 128): 0 = skipped
 * (fully masked), 1 = fully visible, 2 = partial (masked element by element);
 * §18.5.2, Fig. 18-20.  Non-causal shapes answer 1.  -1 on bad arguments. */
int fa_tile_class(const fa_shape_t* shape, int q_tile, int kv_tile);
/* Work units in the order the kernels hand them out (longest first for causal
 * shapes; lecture slides 27-46).  Forward unit = (b, h, pair p: query tiles 2p
 * and 2p+1).  dK/dV unit = (b, kv head, key tile).  dQ unit = (b, h, query
 * tile).  *_num_units gives the count; *_unit writes the index-th unit. */
int fa_fwd_num_units(const fa_shape_t* shape);
int fa_fwd_unit(const fa_shape_t* shape, int index, int* b, int* h, int* p);
int fa_dkdv_num_units(const fa_shape_t* shape);
int fa_dkdv_unit(const fa_shape_t* shape, int index, int* b, int* kvh, int* kv_tile);
int fa_dq_num_units(const fa_shape_t* shape);
int fa_dq_unit(const fa_shape_t* shape, int index, int* b, int* h, int* q_tile);
/* The static schedule of a causal bf16 forward on `grid` CTAs (the launch uses
 * grid = min(units, SMs)): CTA c runs units ord[start[c] .. start[c+1]) in that
 * order.  A causal unit's cost grows with its query tiles, so instead of handing
 * units out longest first from a counter, the host assigns them once per shape:
 * longest first onto the least loaded CTA, then moves and swaps that lower the
 * largest load (cost = the unit's 128 x 128 x d products plus a fixed cost per
 * unit measured on GB300).  start: grid + 1 ints, ord: fa_fwd_num_units ints.
 * FA_ERR_INVALID when the forward does not use one (not causal, more than 2048
 * units or 160 CTAs); it then claims units from a counter, longest first. */
int fa_fwd_schedule(const fa_shape_t* shape, int grid, int* start, int* ord);
/* The key-split plan of an unmasked bf16 forward on `sms` SMs: units split0 ..
 * fa_fwd_num_units - 1 (those of the last, partial wave; all units when there are
 * fewer than SMs) each run as *nsplit parts of whole key tiles, part k covering
 * key tiles [k n / nsplit, (k + 1) n / nsplit) of the n = ceil(Nk / 128), and a
 * combine merges the parts by their LSE.  *nsplit = 1 (and *split0 = the unit
 * count): no split.  The rule: R = U mod sms (U when U < sms) units in the last
 * wave, nsplit = min(floor(sms / R), 4, floor(n / 2)), used when at least 2.
 * FA_ERR_INVALID for a masked (causal or windowed) shape: those never split. */
int fa_fwd_split_plan(const fa_shape_t* shape, int sms, int* split0, int* nsplit);
/* Key range [start, end) of decode split s. */
int fa_decode_split_range(const fa_shape_t* shape, int num_splits, int s, int* start, int* end);

/* ---------------------------------------------------------------------------
 * Diagnostics: one 128-row tcgen05 matrix product through the same TMA,
 * descriptor and TMEM code the attention kernels use (no counterpart on the
 * pages; it isolates the tensor-core building blocks).
 *   mode 0: c[128 x 128] = a[128 x k] * b[128 x k]^T   (both K-major, k = 64|128)
 *   mode 1: c[128 x n]   = a[128 x 128] * b[128 x n]   (a staged in TMEM,
 *                                                       b row-major, n = 64|128)
 *   modes 2, 3: the forms of modes 0 and 1 with E4M3 operands (one-byte codes,
 *           k = n = 128), as the FP8 forward uses them.
 * a, b: device bf16 (modes 0, 1) or E4M3 codes (modes 2, 3), row-major;
 * c: device fp32 row-major.
 * workspace: at least 256 bytes of device memory (its first word records a
 * timed-out wait, as for the attention calls).
 */
int fa_selftest_mma(int mode, int n_or_k, const void* a, const void* b, float* c, void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
