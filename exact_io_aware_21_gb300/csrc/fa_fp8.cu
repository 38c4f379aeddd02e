// E4M3 quantiser for the FP8 forward ("第18章 FlashAttention" §18.6.2, part 2;
// incoherent processing: "CMU 11-868 L21" notes, slide 24).
//
// X_fp8 = E4M3(X / s) with s = max|X| / 448 over a block: 128 rows of one head
// (the forward's load block; Q and K), or every row of one head (V).  With a
// sign vector the rows are first rotated by J = diag(signs) H_d / sqrt(d): the
// unnormalised Walsh-Hadamard transform runs in registers (radix-2 butterflies
// at strides 1, 2, ..., d/2), the codes come from it directly (the block scale
// absorbs any constant factor), and 1 / sqrt(d) goes into the scale.
//
// One CTA of 128 threads per block of rows, thread = row (rows staged through
// shared memory with coalesced loads and stores).  Every rounding that
// decides a code is an IEEE round-to-nearest fp32 operation (sums, 448 / amax,
// y * inv) followed by the hardware's round-to-nearest-even E4M3 conversion, so
// the codes are reproducible operation by operation.  HBM-bound: 2 bytes read
// and 1 written per element (per-head scales read the rows twice).
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float E4M3_MAX = 448.f;

// Shared-memory staging: the block's rows are loaded and stored with coalesced
// 16-byte accesses (a warp covers whole rows), and each thread works on one row
// from shared memory.  Row pitch padded by 16 bytes so that the row-per-thread
// accesses of a quarter warp fall in distinct banks.
template <int D>
struct QuantSmem {
  static constexpr int IN_PITCH = D * 2 + 16;   // bf16 row
  static constexpr int OUT_PITCH = D + 16;      // code row
  static constexpr int BYTES = 128 * IN_PITCH + 128 * OUT_PITCH;
};

template <int D, bool HAD, int MODE>  // MODE 0: block scales; 1: per-head max pass; 2: per-head codes
__global__ void __launch_bounds__(128) quantize_kernel(const QuantLaunch p) {
  using S = QuantSmem<D>;
  extern __shared__ __align__(16) uint8_t qsm[];
  uint8_t* s_in = qsm;
  uint8_t* s_out = qsm + 128 * S::IN_PITCH;
  __shared__ float s_signs[D];
  __shared__ float s_red[4];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n0 = blk * 128;
  const int rows = min(128, p.N - n0);
  if (HAD)
    for (int i = threadIdx.x; i < D; i += 128) s_signs[i] = p.signs[i];

  // coalesced load of the block: chunk c = (row, 16-byte piece)
  constexpr int CPR = D * 2 / 16;  // 16-byte chunks per bf16 row
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(p.x) + b * p.sb + h * p.sh;
#pragma unroll
  for (int c = threadIdx.x; c < 128 * CPR; c += 128) {  // all of a thread's loads in flight at once
    const int r = c / CPR, q = c % CPR;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (r < rows) w = *reinterpret_cast<const uint4*>(xb + static_cast<int64_t>(n0 + r) * p.sn + q * 8);
    *reinterpret_cast<uint4*>(s_in + r * S::IN_PITCH + q * 16) = w;
  }
  __syncthreads();

  const int r = threadIdx.x;
  float y[D];
#pragma unroll
  for (int q = 0; q < D / 8; ++q) {
    const uint4 w = *reinterpret_cast<const uint4*>(s_in + r * S::IN_PITCH + q * 16);
    const float2 a = unpack_bf16(w.x), bb = unpack_bf16(w.y), c = unpack_bf16(w.z), d = unpack_bf16(w.w);
    y[8 * q + 0] = a.x;
    y[8 * q + 1] = a.y;
    y[8 * q + 2] = bb.x;
    y[8 * q + 3] = bb.y;
    y[8 * q + 4] = c.x;
    y[8 * q + 5] = c.y;
    y[8 * q + 6] = d.x;
    y[8 * q + 7] = d.y;
  }
  if (HAD) {
#pragma unroll
    for (int i = 0; i < D; ++i) y[i] *= s_signs[i];  // exact: a sign flip
#pragma unroll
    for (int hs = 1; hs < D; hs *= 2) {
#pragma unroll
      for (int i = 0; i < D; ++i) {
        if (i & hs) continue;
        const float u = y[i], v = y[i + hs];
        y[i] = __fadd_rn(u, v);
        y[i + hs] = __fsub_rn(u, v);
      }
    }
  }

  float amax;
  if (MODE == 2) {
    amax = __uint_as_float(p.head_amax[static_cast<int64_t>(b) * p.H + h]);
  } else {
    float am = 0.f;  // rows past N were loaded as zeros
#pragma unroll
    for (int i = 0; i < D; ++i) am = fmaxf(am, fabsf(y[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = am;
    __syncthreads();
    amax = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
    if (MODE == 1) {  // non-negative floats order like their bit patterns
      if (threadIdx.x == 0) atomicMax(p.head_amax + static_cast<int64_t>(b) * p.H + h, __float_as_uint(amax));
      return;
    }
  }

  const float inv = amax > 0.f ? __fdiv_rn(E4M3_MAX, amax) : 0.f;
#pragma unroll
  for (int q = 0; q < D / 16; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 16 * q + 4 * e;
      w[e] = pack4_e4m3(__fmul_rn(y[i], inv), __fmul_rn(y[i + 1], inv), __fmul_rn(y[i + 2], inv),
                        __fmul_rn(y[i + 3], inv));
    }
    *reinterpret_cast<uint4*>(s_out + r * S::OUT_PITCH + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  constexpr int CPO = D / 16;  // 16-byte chunks per code row
  uint8_t* ob = static_cast<uint8_t*>(p.out) + b * p.ob + h * p.oh;
#pragma unroll 4
  for (int c = threadIdx.x; c < rows * CPO; c += 128) {
    const int rr = c / CPO, q = c % CPO;
    *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(n0 + rr) * p.on + q * 16) =
        *reinterpret_cast<const uint4*>(s_out + rr * S::OUT_PITCH + q * 16);
  }
  if (threadIdx.x == 0 && (MODE == 0 || blk == 0)) {
    float sc = amax > 0.f ? __fdiv_rn(amax, E4M3_MAX) : 0.f;
    if (HAD) sc = __fmul_rn(sc, D == 128 ? 0.0883883476483184405f : 0.125f);  // 1 / sqrt(d)
    const int64_t bh = static_cast<int64_t>(b) * p.H + h;
    p.scales[MODE == 0 ? bh * p.nblk + blk : bh] = sc;
  }
}

template <int D, bool HAD, int MODE>
cudaError_t launch_quantize_mode(const QuantLaunch& a, cudaStream_t st) {
  const dim3 grid(a.nblk, a.H, a.B);
  auto kern = quantize_kernel<D, HAD, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QuantSmem<D>::BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, QuantSmem<D>::BYTES, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool HAD>
cudaError_t launch_quantize_t(const QuantLaunch& a, cudaStream_t st) {
  if (a.per_block) return launch_quantize_mode<D, HAD, 0>(a, st);
  cudaError_t e = launch_quantize_mode<D, HAD, 1>(a, st);
  if (e != cudaSuccess) return e;
  return launch_quantize_mode<D, HAD, 2>(a, st);
}

}  // namespace

cudaError_t launch_quantize(const QuantLaunch& a, cudaStream_t st) {
  const bool had = a.signs != nullptr;
  if (a.d == 64) return had ? launch_quantize_t<64, true>(a, st) : launch_quantize_t<64, false>(a, st);
  return had ? launch_quantize_t<128, true>(a, st) : launch_quantize_t<128, false>(a, st);
}

}  // namespace fa
