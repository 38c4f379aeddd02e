// Work plans of packed variable-length sequences (see plan_unit in fa_plan.h).
//
// The kernels' unit grid is sized by the longest sequence; most of its units
// are empty when lengths vary.  This kernel lists only the units with work,
// longest first across sequences ("CMU 11-868 L21" notes, slides 27-46: hand
// out the longest work first), so no warp role spends a claim on an empty unit.
// One CTA: a counting sort of the sequences by their level count, then the
// level start offsets.  The order of sequences with equal counts follows the
// atomics (it only decides which SM runs which unit, never a result).
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int PLAN_THREADS = 1024;

__device__ __forceinline__ int level_count(const Dims& d, int b, int mode, int* status) {
  const SeqRows sr = seq_rows<true>(d, b);
  if (!sr.ok && status != nullptr) atomicOr(status, FA_STATUS_BAD_INPUT);  // such a sequence gets no units
  if (mode == VARLEN_PLAN_FWD) return cdiv(q_tiles(sr.s), 2);
  if (mode == VARLEN_PLAN_DQ) return q_tiles(sr.s);
  return k_tiles(sr.s);  // dK/dV: every key tile, queries or not
}

__global__ void __launch_bounds__(PLAN_THREADS) varlen_plan_kernel(const Dims d, int mode, int nlev, int heads,
                                                                   int* plan, int* status) {
  extern __shared__ int sh[];
  int* hist = sh;             // [nlev + 1] sequences per level count
  int* cursor = sh + nlev + 1;  // [nlev + 1] next position of each count in the order
  for (int c = threadIdx.x; c <= nlev; c += PLAN_THREADS) hist[c] = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < d.B; b += PLAN_THREADS) atomicAdd(&hist[imin(level_count(d, b, mode, status), nlev)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    // sequences with more levels first: cursor[c] = #sequences with count > c
    int above = 0;
    for (int c = nlev; c >= 0; --c) {
      cursor[c] = above;
      above += hist[c];
    }
    // level v (units of the sequences with count > v), highest first
    int* ls = plan + 4;
    int start = 0;
    for (int k = 0; k < nlev; ++k) {
      const int v = nlev - 1 - k;
      ls[k] = start;
      start += cursor[v] * heads;
    }
    ls[nlev] = start;
    plan[0] = start;
    plan[1] = nlev;
  }
  __syncthreads();
  int* order = plan + 4 + nlev + 1;
  for (int b = threadIdx.x; b < d.B; b += PLAN_THREADS) order[atomicAdd(&cursor[imin(level_count(d, b, mode, nullptr), nlev)], 1)] = b;
}

}  // namespace

cudaError_t launch_varlen_plan(const Dims& d, int mode, int nlev, int heads, int* plan, int* status,
                               cudaStream_t st) {
  const size_t smem = 2 * static_cast<size_t>(nlev + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(varlen_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  varlen_plan_kernel<<<1, PLAN_THREADS, smem, st>>>(d, mode, nlev, heads, plan, status);
  return cudaGetLastError();
}

}  // namespace fa
