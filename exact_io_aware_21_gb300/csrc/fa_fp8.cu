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
// Persistent CTAs of 128 threads stream 128-row blocks, thread = row, the next
// block's TMA load overlapping the current block's work.  Every rounding that
// decides a code is an IEEE round-to-nearest fp32 operation (sums, 448 / amax,
// y * inv) followed by the hardware's round-to-nearest-even E4M3 conversion, so
// the codes are reproducible operation by operation.  HBM-bound: 2 bytes read
// and 1 written per element (per-head scales read the rows twice).
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float E4M3_MAX = 448.f;

// A persistent CTA streams 128-row blocks through two shared-memory stages:
// the TMA load of the next block (64-column boxes, 128-byte swizzle) is in
// flight while all threads transform and encode the current one, thread = row.
// Two stages leave room for three CTAs per SM, whose interleaving hides more
// of the per-block latency than a deeper ring in fewer CTAs (measured).  Once every row is in registers the block's codes are written over its
// own stage (row pitch padded by 16 bytes: the row-per-thread writes of a
// quarter warp fall in distinct banks) and stored with coalesced 16-byte writes.
template <int D>
struct QuantSmem {
  static constexpr int STAGES = 2;
  static constexpr int BOX = 128 * 128;        // one 64-column box of 128 rows (bytes)
  static constexpr int STAGE = D * 2 * 128;    // a block of bf16 rows: D / 64 boxes
  static constexpr int OUT_PITCH = D + 16;     // code row (written over the stage)
  static_assert(128 * OUT_PITCH <= STAGE, "codes fit in their stage");
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int BYTES = OFF_BAR + 64;
  static constexpr int ALLOC = BYTES + 1024;   // 1024-byte alignment of the stages
};

template <int D, bool HAD, int MODE>  // MODE 0: block scales; 1: per-head max pass; 2: per-head codes
__global__ void __launch_bounds__(128) quantize_kernel(const __grid_constant__ CUtensorMap tm_x, const QuantLaunch p) {
  using S = QuantSmem<D>;
  extern __shared__ __align__(1024) uint8_t qraw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qraw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);  // [STAGES]
  __shared__ float s_signs[D];
  __shared__ float s_red[4];
  const Ctl ctl{p.status, p.timeout_ns};
  const int total = p.B * p.H * p.nblk;
  const int r = threadIdx.x;
  if (HAD)
    for (int i = r; i < D; i += 128) s_signs[i] = p.signs[i];
  if (r == 0) {
    for (int k = 0; k < S::STAGES; ++k) mbar_init(&full[k], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_x);
  }
  __syncthreads();
  auto issue = [&](int unit, int stage) {  // unit = (b * H + h) * nblk + blk
    const int blk = unit % p.nblk, bh = unit / p.nblk;
    mbar_arrive_expect_tx(&full[stage], S::STAGE);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_4d(smem + stage * S::STAGE + c * S::BOX, &tm_x, &full[stage], c * 64, bh % p.H, blk * 128, bh / p.H);
  };
  if (r == 0)
    for (int k = 0; k < S::STAGES - 1; ++k)
      if (static_cast<int>(blockIdx.x + k * gridDim.x) < total) issue(blockIdx.x + k * gridDim.x, k);

  int i = 0;
  for (int unit = blockIdx.x; unit < total; unit += gridDim.x, ++i) {
    const int st = i % S::STAGES;
    const int ahead = unit + (S::STAGES - 1) * gridDim.x;
    // that stage held the block before this one, released at the end of the last iteration
    if (r == 0 && ahead < total) issue(ahead, (i + S::STAGES - 1) % S::STAGES);
    const bool ok = mbar_wait(&full[st], (i / S::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_LOAD);
    if (!__syncthreads_and(ok)) break;
    const int blk = unit % p.nblk, bh = unit / p.nblk, b = bh / p.H, h = bh % p.H;
    const int rows = min(128, p.N - blk * 128);  // rows past N were read as zeros

    // this thread's row, un-swizzled: 16-byte chunk c of a box row sits at chunk c ^ (row & 7)
    float y[D];
    const uint8_t* in = smem + st * S::STAGE + r * 128;
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
      const uint4 w = *reinterpret_cast<const uint4*>(in + (q / 8) * S::BOX + (((q % 8) ^ (r & 7)) << 4));
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
    if (HAD) {  // the same IEEE operations as the scalar transform, two lanes at a time where they pair up
#pragma unroll
      for (int k = 0; k < D; k += 2) {  // exact: a sign flip
        const float2 v = __fmul2_rn(make_float2(y[k], y[k + 1]), make_float2(s_signs[k], s_signs[k + 1]));
        y[k] = v.x;
        y[k + 1] = v.y;
      }
#pragma unroll
      for (int k = 0; k < D; k += 2) {  // stride 1: the pair is (y[k], y[k+1])
        const float u = y[k], v = y[k + 1];
        y[k] = __fadd_rn(u, v);
        y[k + 1] = __fsub_rn(u, v);
      }
#pragma unroll
      for (int hs = 2; hs < D; hs *= 2) {  // strides >= 2: (y[k], y[k+1]) against (y[k+hs], y[k+hs+1])
#pragma unroll
        for (int k = 0; k < D; k += 2) {
          if (k & hs) continue;
          const float2 u = make_float2(y[k], y[k + 1]), v = make_float2(y[k + hs], y[k + hs + 1]);
          const float2 sum = __fadd2_rn(u, v);
          const float2 dif = __fadd2_rn(u, make_float2(-v.x, -v.y));  // u - v, exactly
          y[k] = sum.x;
          y[k + 1] = sum.y;
          y[k + hs] = dif.x;
          y[k + hs + 1] = dif.y;
        }
      }
    }

    float amax;
    if (MODE == 2) {
      amax = __uint_as_float(p.head_amax[static_cast<int64_t>(b) * p.H + h]);
    } else {
      float am = 0.f;
#pragma unroll
      for (int k = 0; k < D; k += 2) am = fmax3(am, fabsf(y[k]), fabsf(y[k + 1]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      if ((r & 31) == 0) s_red[r >> 5] = am;
      __syncthreads();
      amax = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
    }
    if (MODE == 1) {  // non-negative floats order like their bit patterns
      if (r == 0) atomicMax(p.head_amax + static_cast<int64_t>(b) * p.H + h, __float_as_uint(amax));
    } else {
      uint8_t* s_out = smem + st * S::STAGE;  // the codes go over the rows just read
      if (MODE == 2) __syncthreads();         // (blocks with a max already synchronised after reading)
      const float inv = amax > 0.f ? __fdiv_rn(E4M3_MAX, amax) : 0.f;
#pragma unroll
      for (int q = 0; q < D / 16; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 16 * q + 4 * e;
          const float2 a = __fmul2_rn(make_float2(y[k], y[k + 1]), make_float2(inv, inv));
          const float2 c = __fmul2_rn(make_float2(y[k + 2], y[k + 3]), make_float2(inv, inv));
          w[e] = pack4_e4m3(a.x, a.y, c.x, c.y);
        }
        *reinterpret_cast<uint4*>(s_out + r * S::OUT_PITCH + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      __syncthreads();
      constexpr int CPO = D / 16;  // 16-byte chunks per code row
      uint8_t* ob = static_cast<uint8_t*>(p.out) + b * p.ob + h * p.oh;
#pragma unroll 4
      for (int c = r; c < rows * CPO; c += 128) {
        const int rr = c / CPO, q = c % CPO;
        *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(blk * 128 + rr) * p.on + q * 16) =
            *reinterpret_cast<const uint4*>(s_out + rr * S::OUT_PITCH + q * 16);
      }
      if (r == 0 && (MODE == 0 || blk == 0)) {
        float sc = amax > 0.f ? __fdiv_rn(amax, E4M3_MAX) : 0.f;
        if (HAD) sc = __fmul_rn(sc, D == 128 ? 0.0883883476483184405f : 0.125f);  // 1 / sqrt(d)
        const int64_t bhi = static_cast<int64_t>(b) * p.H + h;
        p.scales[MODE == 0 ? bhi * p.nblk + blk : bhi] = sc;
      }
    }
    // The code rows were written over the stage through the generic proxy; a later
    // TMA load (async proxy) refills it, so order those writes before it.
    if (MODE != 1) fence_proxy_async_smem();
    __syncthreads();  // the stage, the code rows and s_red are free for the next block
  }
  // loads issued for blocks this CTA gave up on must land before exit
  if (r == 0) {
    const int n_issued = total > static_cast<int>(blockIdx.x)
                             ? (total - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    for (int k = i; k < n_issued && k < i + S::STAGES; ++k)
      mbar_wait(&full[k % S::STAGES], (k / S::STAGES) & 1, ctl, FA_STATUS_TIMEOUT_DRAIN);
  }
}

template <int D, bool HAD, int MODE>
cudaError_t launch_quantize_mode(const QuantLaunch& a, cudaStream_t st) {
  auto kern = quantize_kernel<D, HAD, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QuantSmem<D>::ALLOC);
  if (e != cudaSuccess) return e;
  const int total = a.B * a.H * a.nblk;
  kern<<<imax(1, imin(total, 3 * a.num_sms)), 128, QuantSmem<D>::ALLOC, st>>>(a.tm_x, a);
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
