// quant.cu -- 8-bit (FP8 e4m3) copies of Q and K for the attention's score
// product (MiniAcc blog, "What is SageAttention?": the score computation in
// 8-bit arithmetic). Per (batch, head, 64-token block) of Q and of K:
//   e     = the smallest integer with amax / 2^e <= 448 (0 for an all-zero
//           block), amax = max |x| over the block's valid tokens and all D;
//   code  = x / 2^e rounded to the nearest e4m3 value, ties to even.
// The scale is a power of two, so x / 2^e is exact and the rounding is the
// only approximation; the attention kernel multiplies each logit back by
// 2^(e_q + e_k). Memory-bound: one read of Q and K, one write of the codes.
#include <cmath>
#include <cuda_fp8.h>

#include "sa_internal.cuh"

namespace sa {
namespace {

constexpr int kQuantThreads = 256;

// grid (Nb, H, 2 B): blockIdx.z = 2 b + (0: Q, 1: K); 256 threads, D = 128.
// Thread t handles d-chunk t % 16 (8 values) of tokens t / 16 + 16 p, p < 4.
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(QuantArgs a) {
  constexpr int D = 128, kChunks = D / 8;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, which = blockIdx.z & 1;
  const uint16_t* x = which ? a.k : a.q;
  const int64_t* xs = which ? a.ks : a.qs;
  uint8_t* y = which ? a.k8 : a.q8;
  int8_t* ye = which ? a.k_exp : a.q_exp;
  const int c = threadIdx.x % kChunks, t0 = j * kBlock + threadIdx.x / kChunks;
  __shared__ float warp_max[kQuantThreads / 32];
  __shared__ int block_exp;

  float f[4][8];
  float amax = 0.f;
  bool bad = false;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int t = t0 + 16 * p;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (t < a.S)
      w = __ldg(reinterpret_cast<const uint4*>(x + b * xs[0] + static_cast<int64_t>(t) * xs[1] +
                                               h * xs[2] + 8 * c));
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t word = (&w.x)[u >> 1];
      f[p][u] = __uint_as_float((u & 1) ? (word & 0xffff0000u) : (word << 16));
      const float ax = fabsf(f[p][u]);
      bad |= !(ax <= 3.0e38f);           // inf or NaN
      amax = fmaxf(amax, ax);
    }
  }
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kQuantThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    int e = 0;
    if (m > 0.f && m <= 3.0e38f) {
      // m = fr 2^k with fr in [0.5, 1); 448 = 0.875 * 2^9
      int k = 0;
      const float fr = frexpf(m, &k);
      e = k - 9 + (fr > 0.875f ? 1 : 0);
    }
    block_exp = e;
    ye[(static_cast<int64_t>(b) * a.H + h) * a.Nb + j] = static_cast<int8_t>(e);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && a.dev_status) atomicOr(a.dev_status, SA_DEV_RANGE);
  const int e = block_exp;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int t = t0 + 16 * p;
    if (t >= a.S) continue;
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
      // exact power-of-two scaling, then one rounding to e4m3 (ties to even)
      const float2 v = make_float2(ldexpf(f[p][u], -e), ldexpf(f[p][u + 1], -e));
      const uint32_t pair = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
      if (u < 4) lo |= pair << (8 * u);
      else hi |= pair << (8 * (u - 4));
    }
    *reinterpret_cast<uint2*>(y + b * a.y_stride[0] + static_cast<int64_t>(t) * a.y_stride[1] +
                              h * a.y_stride[2] + 8 * c) = make_uint2(lo, hi);
  }
}

}  // namespace

cudaError_t launch_quant(const QuantArgs& a, cudaStream_t st) {
  dim3 grid(a.Nb, a.H, 2 * a.B);
  quant_kernel<<<grid, kQuantThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
