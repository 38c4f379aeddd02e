// Block-sparse tables for the backward ("第18章 FlashAttention" §18.8.1): the
// caller's CSR table (key tiles per query tile) is checked and filtered once
// per call into the lists the two backward kernels walk:
//   rows:    per query tile, its key tiles in ascending order (dQ)
//   columns: per key tile, the query tiles listing it, ascending (dK/dV)
// and into the dK/dV kernel's segment plan (fa_kernels.h).  Entries out of
// order or out of range are skipped and reported; under j <= i tiles above the
// diagonal are dropped (they hide every key).  Both lists come from a tile
// bitmap scanned in index order and the plan from their lengths alone, so the
// order a kernel sums its tiles in, and therefore every result, is the same on
// every call.
//
// One CTA of 1024 threads does it all with the bitmap in shared memory (one
// bit per tile pair: at most 1024 x 1024 bits = 128 KB): thread i counts row i
// and column i, block-wide scans give the list offsets, thread i writes row
// i's and column i's list.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int LIST_THREADS = 1024;

struct Seg {
  int kt, k0, n, slot;
};

// Exclusive block-wide prefix sum of v over the 1024 threads; *total gets the sum.
// `tmp` holds 32 ints of shared memory; every thread must call it.
__device__ __forceinline__ int block_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    tmp[lane] = t;  // inclusive sums of the warps
  }
  __syncthreads();
  const int r = x - v + (warp > 0 ? tmp[warp - 1] : 0);
  *total = tmp[31];
  __syncthreads();  // tmp is free again
  return r;
}

__global__ void __launch_bounds__(LIST_THREADS) sparse_lists_kernel(SparseLaunch a) {
  extern __shared__ uint32_t bits[];  // [nqt][W]
  __shared__ int tmp[32];
  __shared__ Seg seg[SP_MAX_SEGMENTS];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = (a.nkt + 31) >> 5;
  for (int i = tid; i < a.nqt * W; i += LIST_THREADS) bits[i] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // 1) mark: one warp per query tile at a time
  for (int qt = warp; qt < a.nqt; qt += LIST_THREADS / 32) {
    const int e0 = __ldg(a.row_ptr + qt), e1 = __ldg(a.row_ptr + qt + 1);
    bool bad = e0 < 0 || e1 < e0 || e1 > a.nnz;
    if (!bad) {
      for (int e = e0 + lane; e < e1; e += 32) {
        const int c = __ldg(a.col_idx + e);
        const int prev = e > e0 ? __ldg(a.col_idx + e - 1) : -1;
        if (c <= prev || c < 0 || c >= a.nkt) {
          bad = true;
          continue;
        }
        if (a.causal && c > qt) continue;
        atomicOr(&bits[qt * W + (c >> 5)], 1u << (c & 31));
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) s_bad = 1;
  }
  __syncthreads();
  if (tid == 0 && s_bad) atomicOr(a.status, FA_STATUS_BAD_INPUT);

  // 2) counts and offsets
  int rc = 0, cc = 0;
  if (tid < a.nqt)
    for (int w = 0; w < W; ++w) rc += __popc(bits[tid * W + w]);
  if (tid < a.nkt)
    for (int r = 0; r < a.nqt; ++r) cc += (bits[r * W + (tid >> 5)] >> (tid & 31)) & 1;
  int rtot, ctot;
  const int roff = block_scan(rc, tmp, &rtot);
  const int coff = block_scan(cc, tmp, &ctot);
  if (tid < a.nqt) a.rows_ptr[tid] = roff;
  if (tid < a.nkt) a.cols_ptr[tid] = coff;
  if (tid == 0) {
    a.rows_ptr[a.nqt] = rtot;
    a.cols_ptr[a.nkt] = ctot;
  }

  // 3) the lists, ascending
  if (tid < a.nqt) {
    int w = roff;
    for (int x = 0; x < W; ++x) {
      uint32_t m = bits[tid * W + x];
      while (m) {
        a.rows_idx[w++] = x * 32 + __ffs(m) - 1;
        m &= m - 1;
      }
    }
  }
  if (tid < a.nkt) {
    int w = coff;
    for (int r = 0; r < a.nqt; ++r)
      if ((bits[r * W + (tid >> 5)] >> (tid & 31)) & 1) a.cols_idx[w++] = r;
  }

  // 4) the dK/dV plan.  n = this key tile's iterations; W_total = heads x sum(n);
  // seg = max(SP_MIN_SEGMENT, ceil(W_total / SP_PLAN_PARALLELISM)).  A split
  // tile has ceil(n / seg) < 2 n / seg segments and sum(n) / seg <= P / heads,
  // so a head group has fewer than nkt + 2P segments and all heads together
  // fewer than min(2P, W_total / 16) slots: the plan and the pool always fit
  // (checked all the same: a plan that would not fit is built unsplit).
  const int n = tid < a.nkt ? a.group * cc : 0;
  int ntot;
  block_scan(n, tmp, &ntot);
  const long long wtot = static_cast<long long>(a.heads) * ntot;
  long long segl = (wtot + SP_PLAN_PARALLELISM - 1) / SP_PLAN_PARALLELISM;
  if (segl < SP_MIN_SEGMENT) segl = SP_MIN_SEGMENT;
  int seg_len = segl > 0x40000000LL ? 0x40000000 : static_cast<int>(segl);
  int ns = 0, slots = 0, nsplit = 0, soff = 0, sloff = 0, spoff = 0, nseg = 0;
  for (int pass = 0; pass < 2; ++pass) {
    nseg = tid < a.nkt ? (n > seg_len ? (n + seg_len - 1) / seg_len : 1) : 0;
    soff = block_scan(nseg, tmp, &ns);
    sloff = block_scan(nseg > 1 ? nseg : 0, tmp, &slots);
    spoff = block_scan(nseg > 1 ? 1 : 0, tmp, &nsplit);
    if (ns <= SP_MAX_SEGMENTS && static_cast<long long>(slots) * a.heads <= a.pool_slots) break;
    seg_len = 0x40000000;  // unreachable by the bound above; keep every tile whole
  }
  if (tid < a.nkt) {
    const int base = n / nseg, extra = n % nseg;
    for (int s = 0; s < nseg; ++s)
      seg[soff + s] = Seg{tid, s * base + (s < extra ? s : extra), base + (s < extra ? 1 : 0),
                          nseg > 1 ? sloff + s : -1};
    if (nseg > 1) {
      int4* sp = reinterpret_cast<int4*>(a.dkdv_plan + SP_PLAN_SPLITS) + spoff;
      *sp = make_int4(tid, sloff, nseg, 0);
    }
  }
  __syncthreads();
  // longest first; equal lengths keep their (key tile, first iteration) order
  int4* out = reinterpret_cast<int4*>(a.dkdv_plan + SP_PLAN_SEGS);
  for (int i = tid; i < ns; i += LIST_THREADS) {
    const Seg e = seg[i];
    int rank = 0;
    for (int j = 0; j < ns; ++j) {
      const int nj = seg[j].n;
      rank += (nj > e.n) || (nj == e.n && j < i);
    }
    out[rank] = make_int4(e.kt, e.k0, e.n, e.slot);
  }
  if (tid == 0) {
    a.dkdv_plan[0] = ns;
    a.dkdv_plan[1] = slots;
    a.dkdv_plan[2] = nsplit;
    a.dkdv_plan[3] = seg_len;
  }
}

size_t sparse_lists_smem(int nqt, int nkt) { return static_cast<size_t>(nqt) * ((nkt + 31) / 32) * 4; }

}  // namespace

cudaError_t launch_sparse_lists(const SparseLaunch& a, cudaStream_t st) {
  if (a.nqt > LIST_THREADS || a.nkt > LIST_THREADS || a.nqt < 1 || a.nkt < 1) return cudaErrorInvalidValue;
  const size_t smem = sparse_lists_smem(a.nqt, a.nkt);
  cudaError_t e = cudaFuncSetAttribute(sparse_lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  sparse_lists_kernel<<<1, LIST_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
