// Block-sparse tables for the backward ("第18章 FlashAttention" §18.8.1): the
// caller's CSR table (key tiles per query tile) is checked and filtered once
// per call into the lists the two backward kernels walk:
//   rows:    per query tile, its key tiles in ascending order (dQ)
//   columns: per key tile, the query tiles listing it, ascending (dK/dV)
// Entries out of order or out of range are skipped and reported; under j <= i
// tiles above the diagonal are dropped (they hide every key).  Both lists come
// from a tile bitmap scanned in index order, so the order a kernel sums its
// tiles in, and therefore every result, is the same on every call.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int LIST_THREADS = 1024;

// One warp per query tile: mark the tiles its row lists.
__global__ void __launch_bounds__(32) sparse_mark_kernel(SparseLaunch a) {
  const int qt = blockIdx.x, lane = threadIdx.x;
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
      a.bitmap[static_cast<int64_t>(qt) * a.nkt + c] = 1;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, FA_STATUS_BAD_INPUT);
}

// One CTA: thread i counts row i and column i of the bitmap, the counts are
// prefix-summed, and each thread writes its row's and its column's list.
__global__ void __launch_bounds__(LIST_THREADS) sparse_lists_kernel(SparseLaunch a) {
  __shared__ int s_row[LIST_THREADS + 1], s_col[LIST_THREADS + 1];
  const int i = threadIdx.x;
  int rc = 0, cc = 0;
  if (i < a.nqt)
    for (int c = 0; c < a.nkt; ++c) rc += a.bitmap[static_cast<int64_t>(i) * a.nkt + c];
  if (i < a.nkt)
    for (int r = 0; r < a.nqt; ++r) cc += a.bitmap[static_cast<int64_t>(r) * a.nkt + i];
  s_row[i + 1] = rc;
  s_col[i + 1] = cc;
  if (i == 0) s_row[0] = s_col[0] = 0;
  __syncthreads();
  if (i == 0) {
    for (int k = 1; k <= LIST_THREADS; ++k) {
      s_row[k] += s_row[k - 1];
      s_col[k] += s_col[k - 1];
    }
  }
  __syncthreads();
  if (i < a.nqt) a.rows_ptr[i] = s_row[i];
  if (i < a.nkt) a.cols_ptr[i] = s_col[i];
  if (i == 0) {
    a.rows_ptr[a.nqt] = s_row[a.nqt];
    a.cols_ptr[a.nkt] = s_col[a.nkt];
  }
  if (i < a.nqt) {
    int w = s_row[i];
    for (int c = 0; c < a.nkt; ++c)
      if (a.bitmap[static_cast<int64_t>(i) * a.nkt + c]) a.rows_idx[w++] = c;
  }
  if (i < a.nkt) {
    int w = s_col[i];
    for (int r = 0; r < a.nqt; ++r)
      if (a.bitmap[static_cast<int64_t>(r) * a.nkt + i]) a.cols_idx[w++] = r;
  }
}

}  // namespace

cudaError_t launch_sparse_lists(const SparseLaunch& a, cudaStream_t st) {
  if (a.nqt > LIST_THREADS || a.nkt > LIST_THREADS) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.bitmap, 0, static_cast<size_t>(a.nqt) * a.nkt, st);
  if (e != cudaSuccess) return e;
  sparse_mark_kernel<<<a.nqt, 32, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sparse_lists_kernel<<<1, LIST_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
