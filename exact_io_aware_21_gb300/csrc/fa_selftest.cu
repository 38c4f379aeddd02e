// Self-test of the tensor-core building blocks: one 128-row tcgen05 product
// through the same TMA maps, shared-memory descriptors, instruction
// descriptors and TMEM accesses as the attention kernels.
//   mode 0: C[128 x 128] = A[128 x K] B[128 x K]^T   (the S = Q K^T form)
//   mode 1: C[128 x N]   = A[128 x 128] B[128 x N]   (the O += P V form: A is
//           written to TMEM as packed bf16, B is N-major in shared memory)
//   modes 2 and 3: the same two forms with E4M3 operands (kind::f8f6f4), K = N
//           = 128: A and B rows of 128 one-byte codes, A of mode 3 written to
//           TMEM four codes per column.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int mode,
                    int nk, const void* a_rows, float* c, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;                 // 32 KB
  uint8_t* sb = smem + 32768;         // 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 65536);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  const Ctl ctl{status, 2000000000ull};
  const int warp = threadIdx.x >> 5, lane = lane_id();
  const int r = threadIdx.x;  // row = TMEM lane

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);  // loads landed
    mbar_init(&bars[1], 1);  // MMA done
    mbar_init(&bars[2], 128);  // A staged in TMEM
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
  const int ncols = (mode == 0 || mode == 2) ? 128 : nk;
  const bool f8 = mode >= 2;

  if (mode == 3) {  // stage A rows as packed E4M3 quadruples in TMEM columns [0, 32)
    const uint32_t* src = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a_rows) + r * 128);
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = src[i];
    tmem_st32(tmem + lanes, v);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars[2]);
  }
  if (mode == 1) {  // stage A rows as packed bf16 pairs in TMEM columns [0, 64)
    const uint32_t* src = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a_rows) + r * 128);
    uint32_t v[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = src[h * 32 + i];
      tmem_st32(tmem + lanes + h * 32, v);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars[2]);
  }

  if (threadIdx.x == 0) {
    const int esz = f8 ? 1 : 2;                       // bytes per element
    const int ch = nk * esz / 128;                    // 128-byte boxes per row
    const bool a_smem = mode == 0 || mode == 2;
    const uint32_t bytes_a = a_smem ? 128 * nk * esz : 0;
    const uint32_t bytes_b = 128 * nk * esz;
    mbar_arrive_expect_tx(&bars[0], bytes_a + bytes_b);
    for (int q = 0; q < ch; ++q) {
      if (a_smem) tma_load_4d(sa + q * 16384, &tm_a, &bars[0], q * (128 / esz), 0, 0, 0);
      tma_load_4d(sb + q * 16384, &tm_b, &bars[0], q * (128 / esz), 0, 0, 0);
    }
    bool ok = mbar_wait(&bars[0], 0, ctl, FA_STATUS_TIMEOUT_MMA);
    if (mode == 1 || mode == 3) ok = ok && mbar_wait(&bars[2], 0, ctl, FA_STATUS_TIMEOUT_MMA);
    tc_fence_after();
    if (ok) {
      const uint32_t a_base = smem_u32(sa), b_base = smem_u32(sb);
      if (mode == 0) {
        const uint32_t idesc = idesc_bf16(128, 128, false, false);
        for (int k = 0; k < nk / 16; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(tmem + 128, sdesc_sw128(a_base + off, 16, 1024), sdesc_sw128(b_base + off, 16, 1024), idesc,
                 k > 0);
        }
      } else if (mode == 1) {
        const uint32_t idesc = idesc_bf16(128, nk, false, true);
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + 128, tmem + k * 8, sdesc_sw128(b_base + k * 2048, 16384, 1024), idesc, k > 0);
      } else if (mode == 2) {  // K = 128 codes in one 128-byte swizzle row, 32 per product
        const uint32_t idesc = idesc_e4m3(128, 128, false, false);
        for (int k = 0; k < 4; ++k)
          mma_ss_f8(tmem + 128, sdesc_sw128(a_base + k * 32, 16, 1024), sdesc_sw128(b_base + k * 32, 16, 1024),
                    idesc, k > 0);
      } else {  // mode 3: 32 rows of B (one product's K) are 4 swizzle atoms of 8 rows
        const uint32_t idesc = idesc_e4m3(128, 128, false, true);
        for (int k = 0; k < 4; ++k)
          mma_ts_f8(tmem + 128, tmem + k * 8, sdesc_sw128(b_base + k * 32 * 128, 16384, 1024), idesc, k > 0);
      }
      mma_commit(&bars[1]);
    } else {
      mbar_arrive(&bars[1]);
    }
  }
  __syncwarp();
  bool ok = mbar_wait(&bars[1], 0, ctl, FA_STATUS_TIMEOUT_SOFTMAX);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lanes + 128 + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) c[r * ncols + c0 + i] = __uint_as_float(v[i]);
    }
  }
  (void)lane;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_selftest_mma(int mode, int n_or_k, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const void* a_rows, float* c, int* status, cudaStream_t st) {
  const int smem = 65536 + 1024 + 1024;
  cudaError_t e = cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  selftest_kernel<<<1, 128, smem, st>>>(tm_a, tm_b, mode, n_or_k, a_rows, c, status);
  return cudaGetLastError();
}

}  // namespace fa
