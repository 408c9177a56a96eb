// route.cu -- the online block router on sm_103a.
//
// The pages name an online router over compressed (block-pooled) queries
// and keys with threshold tau = 1.0, a diagonal threshold and an exact prefix
// sink ("MiniMax H3 runs on single 4090 with 4.44x speedup over dense
// execution", third paragraph; Sol-Engine H3-DataCenter release page, policy
// paragraph). The rule evaluated here: qbar/kbar = mean of the valid tokens of
// each 64-token block; s_ij = scale * qbar_i . kbar_j over every key block;
// p_ij = softmax_j(s_ij); keep j iff p_ij >= tau/Nb, or j is a sink block
// (j < ceil(P/64)), or j == i. With 128-token query blocks (q_block = 128)
// qbar_i pools query tokens [128 i, 128 i + 128), the diagonal is key blocks
// 2i and 2i + 1, and rows 2i and 2i + 1 of the CSR both get query block i's
// list; the kernels below index routed rows by query block (B*H*Nq of them)
// and only scan/emit expand them to the CSR's B*H*Nb rows.
//
// Kernels, in launch order:
//   pool     Q and K read once; block sums accumulated error-free (TwoSum in
//            fp32, so the fp64 mean is exact to fp64 rounding); writes fp32
//            and fp64 pooled vectors and their 2-norms.          HBM-bound.
//   score    pooled Q . pooled K^T per head, 64x64 fp32 SIMT tiles; writes
//            the logits and each tile's row max / sum of exponentials.
//   select   per row: log-sum-exp from the tile partials, threshold test in
//            log space, forced blocks, a bitmask and a count. A row with a
//            decision inside the fp32 error bound is queued for recheck.
//   recheck  queued rows recomputed wholly in fp64 from the fp64 pooled
//            vectors (the same formula as the definition).
// (prologue: QK-norm + RoPE with the pooling fused in, in place of pool, for
// sa_qk_prologue; sa_route_pooled then runs the kernels from score on.)
//   scan     exclusive scan of the counts -> row_ptr.
//   emit     bitmask -> ascending col_idx, bounded by col_cap.
#include <cfloat>
#include <cmath>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "sa_internal.cuh"

namespace sa {

namespace {

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Two fp32 lanes in one 64-bit register: IEEE round-to-nearest adds and
// subtracts of each lane, subnormals kept (no flush), so each lane rounds
// exactly as the scalar __fadd_rn / __fsub_rn would.
__device__ __forceinline__ uint64_t add2_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// two_sum on both lanes of a pair (the same operations, lane by lane)
__device__ __forceinline__ void two_sum2(uint64_t& s, uint64_t& e, uint64_t b) {
  const uint64_t a = s;
  const uint64_t t = add2_rn(a, b);
  const uint64_t bb = sub2_rn(t, a);
  const uint64_t err = add2_rn(sub2_rn(a, sub2_rn(t, bb)), sub2_rn(b, bb));
  s = t;
  e = add2_rn(e, err);
}

// TwoSum: s + e == a + b exactly (round-to-nearest, no overflow).
__device__ __forceinline__ void two_sum(float& s, float& e, float b) {
  const float a = s;
  const float t = __fadd_rn(a, b);
  const float bb = __fsub_rn(t, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(t, bb)), __fsub_rn(b, bb));
  s = t;
  e = __fadd_rn(e, err);
}

template <typename T>
__device__ __forceinline__ T* ws_ptr(char* ws, size_t off) {
  return reinterpret_cast<T*>(ws + off);
}

// ---------------------------------------------------------------- pool ---
// The block sums of a thread's 8 dims (s + c exact, TwoSum) -> the fp64 and
// fp32 block means and the vector's norm bound, in the route workspace.
// Called by every thread of the CTA (the norm is a shuffle over the D/8
// lanes of a head).
template <int D>
__device__ __forceinline__ void store_pooled(const RouteArgs& a, int which, int b, int h, int d,
                                             int i, int nrow, int n, const float* s,
                                             const float* c, bool active) {
  // Block means: fp64 (s + c is the exact block sum) for the recheck, fp32
  // for the scores. Every block but a ragged last one holds a power-of-two
  // count, so the fp64 division is an exact scaling (one multiply) there: the
  // fp64 unit, a small fraction of the fp32 rate on this GPU, is kept to a
  // conversion, an add and a multiply per value.
  float sq = 0.f;
  if (active) {
    const int bh = b * a.H + h;
    const size_t row = static_cast<size_t>(bh) * nrow + i;
    float* p32 = ws_ptr<float>(a.ws, which ? a.L.kbar32 : a.L.qbar32) + row * D + d;
    double* p64 = ws_ptr<double>(a.ws, which ? a.L.kbar64 : a.L.qbar64) + row * D + d;
    const bool pow2 = (n & (n - 1)) == 0;
    const double inv = 1.0 / static_cast<double>(n);    // exact for a power of two
    double m[8];
    float m32[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const double sum = static_cast<double>(s[u]) + static_cast<double>(c[u]);
      m[u] = pow2 ? sum * inv : sum / static_cast<double>(n);
      // the fp32 mean: the sum rounded once to fp32, then the exact scaling
      m32[u] = pow2 ? __fadd_rn(s[u], c[u]) * static_cast<float>(inv) : static_cast<float>(m[u]);
      sq = fmaf(m32[u], m32[u], sq);
    }
    reinterpret_cast<float4*>(p32)[0] = make_float4(m32[0], m32[1], m32[2], m32[3]);
    reinterpret_cast<float4*>(p32)[1] = make_float4(m32[4], m32[5], m32[6], m32[7]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      reinterpret_cast<double2*>(p64)[u] = make_double2(m[2 * u], m[2 * u + 1]);
  }
  // 2-norm of the pooled vector (an upper bound, for the score error bound):
  // the D/8 threads of one head are adjacent lanes. The fp32 sum of squares
  // of the fp32 means is within a relative 16 u of the exact one (u = 2^-24;
  // 8-term chains, a 4-level tree, the means' own rounding), its square root
  // within 9 u; the factor 1 + 4e-6 covers that and its own rounding.
#pragma unroll
  for (int off = D / 16; off >= 1; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  if (active && d == 0) {
    const int bh = b * a.H + h;
    const size_t row = static_cast<size_t>(bh) * nrow + i;
    const float nrm = sqrtf(sq) * (1.0f + 4e-6f);
    ws_ptr<float>(a.ws, which ? a.L.knorm : a.L.qnorm)[row] = nrm;
    if (which) atomicMax(ws_ptr<int>(a.ws, a.L.kmax) + bh, __float_as_int(nrm));
  }
}

// grid (Nb, ceil(H*D / 1024), 2*B), 128 threads; each thread owns 8
// consecutive d of one head (a 16-byte load per token). Query blocks are
// qblk tokens long (Nq of them per head), key blocks 64.
template <int D>
__global__ void __launch_bounds__(128) pool_kernel(RouteArgs a) {
  const int i = blockIdx.x;
  const int which = blockIdx.z & 1;  // 0: Q, 1: K
  const int b = blockIdx.z >> 1;
  const int e0 = (blockIdx.y * 128 + threadIdx.x) * 8;
  const int HD = a.H * D;
  const bool active = e0 < HD;
  const int h = active ? e0 / D : 0;
  const int d = active ? e0 % D : 0;
  const uint16_t* X = which ? a.k : a.q;
  const int64_t* st = which ? a.ks : a.qs;
  const int blk = which ? kBlock : a.qblk;
  const int nrow = which ? a.Nb : a.Nq;   // pooled rows per head
  if (i >= nrow) return;                  // uniform over the CTA
  const int t0 = i * blk;
  const int n = min(blk, a.S - t0);

  // running sums and error terms of the 8 channels as 4 lane pairs
  // (channels 2v, 2v + 1 in pair v), summed with two_sum2
  uint64_t s2[4], c2[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) s2[v] = c2[v] = 0ull;

  if (active) {
    const uint16_t* base = X + b * st[0] + h * st[2] + d + t0 * st[1];
    for (int t = 0; t < n; t += 8) {
      uint4 buf[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (t + u < n) buf[u] = __ldg(reinterpret_cast<const uint4*>(base + (t + u) * st[1]));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (t + u < n) {
          const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            // the two bf16 of the word as fp32 (exact): low half, high half
            const uint64_t x = (static_cast<uint64_t>(w[v] & 0xffff0000u) << 32) | (w[v] << 16);
            two_sum2(s2[v], c2[v], x);
          }
        }
      }
    }
  }
  float s[8], c[8];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    s[2 * v] = __uint_as_float(static_cast<uint32_t>(s2[v]));
    s[2 * v + 1] = __uint_as_float(static_cast<uint32_t>(s2[v] >> 32));
    c[2 * v] = __uint_as_float(static_cast<uint32_t>(c2[v]));
    c[2 * v + 1] = __uint_as_float(static_cast<uint32_t>(c2[v] >> 32));
  }
  store_pooled<D>(a, which, b, h, d, i, nrow, n, s, c, active);
}

// ------------------------------------------------------------ prologue ---
// QK-norm + RoPE with the pooling fused in ("Making MiniMax-H3 up to 9x
// faster on H100s", section "Custom kernels": a fused QK-norm plus RoPE
// kernel). For each token of a (b, h) head vector x [D]:
//   y_d = x_d / sqrt(mean(x^2) + eps) * gamma_d
//   (y_2i, y_2i+1) -> (y_2i cos - y_2i+1 sin, y_2i sin + y_2i+1 cos), angle of
//   (token, pair i) from the caller's tables
// rounded once to bf16 and stored; the rounded values are summed per block
// exactly as pool_kernel sums what it reads, so the pooled means are those
// sa_route would compute from the outputs, and Q and K are not read again.
// Same grid and thread layout as pool_kernel; plain loads (the outputs may
// overwrite the inputs in place).
template <int D>
__global__ void __launch_bounds__(128) prologue_kernel(RouteArgs a, PrologueArgs pa) {
  constexpr int kLanes = D / 8;       // threads of one head vector
  constexpr int kChunk = 64;          // tokens whose rotary rows are staged at once
  constexpr int kT = 8;               // tokens in flight per thread
  // this chunk's rotary rows, [token][pair]: cos, then sin
  __shared__ __align__(16) float tab[2][kChunk][D / 2];
  const int i = blockIdx.x;
  const int which = blockIdx.z & 1;  // 0: Q, 1: K
  const int b = blockIdx.z >> 1;
  const int e0 = (blockIdx.y * 128 + threadIdx.x) * 8;
  const int HD = a.H * D;
  const bool active = e0 < HD;
  const int h = active ? e0 / D : 0;
  const int d = active ? e0 % D : 0;
  const uint16_t* X = which ? a.k : a.q;
  uint16_t* Y = which ? pa.k_out : pa.q_out;
  const int64_t* st = which ? a.ks : a.qs;
  const float* gamma = which ? pa.gamma_k : pa.gamma_q;
  const int blk = which ? kBlock : a.qblk;
  const int nrow = which ? a.Nb : a.Nq;
  if (i >= nrow) return;                  // uniform over the CTA
  const int t0 = i * blk;
  const int n = min(blk, a.S - t0);
  const float inv_d = 1.0f / static_cast<float>(D);   // exact: D is a power of two
  const bool rope = pa.cos != nullptr;

  float g[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) g[u] = 1.f;
  if (active && gamma) {
    const float4 g0 = reinterpret_cast<const float4*>(gamma + d)[0];
    const float4 g1 = reinterpret_cast<const float4*>(gamma + d)[1];
    g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
    g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
  }
  float s[8], c[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) s[u] = c[u] = 0.f;

  const int64_t off = b * st[0] + h * st[2] + d;
  for (int c0 = 0; c0 < n; c0 += kChunk) {
    const int nc = min(kChunk, n - c0);
    if (rope) {
      // stage the chunk's rotary rows (shared by every head of the CTA)
      __syncthreads();                    // the previous chunk's rows are read
      constexpr int kRow4 = D / 8;        // float4 per table row
      const float4* cs4 = reinterpret_cast<const float4*>(pa.cos) +
                          static_cast<size_t>(t0 + c0) * kRow4;
      const float4* sn4 = reinterpret_cast<const float4*>(pa.sin) +
                          static_cast<size_t>(t0 + c0) * kRow4;
      for (int e = threadIdx.x; e < nc * kRow4; e += 128) {
        reinterpret_cast<float4*>(&tab[0][0][0])[e] = cs4[e];
        reinterpret_cast<float4*>(&tab[1][0][0])[e] = sn4[e];
      }
      __syncthreads();
    }
    // the next kT tokens' loads are in flight while these are transformed
    uint4 xb[kT], xn[kT];
    auto load_batch = [&](int t, uint4* dst) {
#pragma unroll
      for (int u = 0; u < kT; ++u)
        dst[u] = (active && t + u < nc)
                     ? *reinterpret_cast<const uint4*>(X + off + (t0 + c0 + t + u) * st[1])
                     : make_uint4(0u, 0u, 0u, 0u);
    };
    load_batch(0, xb);
    for (int t = 0; t < nc; t += kT) {
      if (t + kT < nc) load_batch(t + kT, xn);
#pragma unroll
      for (int u = 0; u < kT; ++u) {
        const uint32_t w[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
        float x[8];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          x[2 * v] = bf16_to_f32(static_cast<uint16_t>(w[v] & 0xffffu));
          x[2 * v + 1] = bf16_to_f32(static_cast<uint16_t>(w[v] >> 16));
        }
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < 8; ++v) ss = fmaf(x[v], x[v], ss);
#pragma unroll
        for (int o = kLanes / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss * inv_d + pa.eps);
        float cv[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
        if (rope && t + u < nc) {
          const float4 c4 = *reinterpret_cast<const float4*>(&tab[0][t + u][d / 2]);
          const float4 s4 = *reinterpret_cast<const float4*>(&tab[1][t + u][d / 2]);
          cv[0] = c4.x; cv[1] = c4.y; cv[2] = c4.z; cv[3] = c4.w;
          sv[0] = s4.x; sv[1] = s4.y; sv[2] = s4.z; sv[3] = s4.w;
        }
        uint32_t packed[4];
        float yr[8];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float y0 = x[2 * v] * r * g[2 * v];
          const float y1 = x[2 * v + 1] * r * g[2 * v + 1];
          const float o0 = fmaf(y0, cv[v], -y1 * sv[v]);
          const float o1 = fmaf(y0, sv[v], y1 * cv[v]);
          const __nv_bfloat162 hb = __floats2bfloat162_rn(o0, o1);
          packed[v] = *reinterpret_cast<const uint32_t*>(&hb);
          yr[2 * v] = bf16_to_f32(static_cast<uint16_t>(packed[v] & 0xffffu));
          yr[2 * v + 1] = bf16_to_f32(static_cast<uint16_t>(packed[v] >> 16));
        }
        if (active && t + u < nc) {
          *reinterpret_cast<uint4*>(Y + off + (t0 + c0 + t + u) * st[1]) =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
#pragma unroll
          for (int v = 0; v < 8; ++v) two_sum(s[v], c[v], yr[v]);
        }
      }
#pragma unroll
      for (int u = 0; u < kT; ++u) xb[u] = xn[u];
    }
  }
  store_pooled<D>(a, which, b, h, d, i, nrow, n, s, c, active);
}

// --------------------------------------------------------------- score ---
// grid (n_ct, n_qt, B*H), 256 threads; a 64x64 tile of pooled logits
// (query blocks x key blocks), 4x4 outputs per thread, D consumed in chunks
// of 32.
template <int D>
__global__ void __launch_bounds__(256) score_kernel(RouteArgs a) {
  constexpr int T = kScoreTile, KC = 32;
  __shared__ __align__(16) float Qs[KC][T];
  __shared__ __align__(16) float Ks[KC][T];
  const int j0 = blockIdx.x * T, i0 = blockIdx.y * T, bh = blockIdx.z;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const float* qb = ws_ptr<float>(a.ws, a.L.qbar32) + static_cast<size_t>(bh) * a.Nq * D;
  const float* kb = ws_ptr<float>(a.ws, a.L.kbar32) + static_cast<size_t>(bh) * a.Nb * D;

  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

  const int lr = tid >> 2, lc = (tid & 3) * 8;  // loader: row, 8 dims
  for (int d0 = 0; d0 < D; d0 += KC) {
    float4 qa = make_float4(0, 0, 0, 0), qb4 = qa, ka = qa, kb4 = qa;
    if (i0 + lr < a.Nq) {
      const float4* src = reinterpret_cast<const float4*>(qb + static_cast<size_t>(i0 + lr) * D + d0 + lc);
      qa = src[0];
      qb4 = src[1];
    }
    if (j0 + lr < a.Nb) {
      const float4* src = reinterpret_cast<const float4*>(kb + static_cast<size_t>(j0 + lr) * D + d0 + lc);
      ka = src[0];
      kb4 = src[1];
    }
    __syncthreads();
    Qs[lc + 0][lr] = qa.x; Qs[lc + 1][lr] = qa.y; Qs[lc + 2][lr] = qa.z; Qs[lc + 3][lr] = qa.w;
    Qs[lc + 4][lr] = qb4.x; Qs[lc + 5][lr] = qb4.y; Qs[lc + 6][lr] = qb4.z; Qs[lc + 7][lr] = qb4.w;
    Ks[lc + 0][lr] = ka.x; Ks[lc + 1][lr] = ka.y; Ks[lc + 2][lr] = ka.z; Ks[lc + 3][lr] = ka.w;
    Ks[lc + 4][lr] = kb4.x; Ks[lc + 5][lr] = kb4.y; Ks[lc + 6][lr] = kb4.z; Ks[lc + 7][lr] = kb4.w;
    __syncthreads();
    // Each chunk of 32 dims is summed as two fresh 16-term FMA chains that
    // are then added to the running total: the rounding error of a score is
    // then bounded by gamma_{16 + D/16 + 3} (not gamma_{D + 3} of a single
    // chain), which keeps the fp64 recheck band narrow.
#pragma unroll
    for (int hh = 0; hh < KC; hh += 16) {
      float t[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) t[r][c] = 0.f;
#pragma unroll 8
      for (int kk = hh; kk < hh + 16; ++kk) {
        const float4 qv = *reinterpret_cast<const float4*>(&Qs[kk][ty * 4]);
        const float4 kv = *reinterpret_cast<const float4*>(&Ks[kk][tx * 4]);
        const float qr[4] = {qv.x, qv.y, qv.z, qv.w};
        const float kc[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) t[r][c] = fmaf(qr[r], kc[c], t[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] += t[r][c];
    }
  }

  float* scores = ws_ptr<float>(a.ws, a.L.scores);
  float* pm = ws_ptr<float>(a.ws, a.L.part_m);
  float* ps = ws_ptr<float>(a.ws, a.L.part_s);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = i0 + ty * 4 + r;
    float sv[4];
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + tx * 4 + c;
      sv[c] = acc[r][c] * a.scale;
      if (j < a.Nb) mx = fmaxf(mx, sv[c]);
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float se = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + tx * 4 + c;
      if (j < a.Nb) se += expf(sv[c] - mx);
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) se += __shfl_xor_sync(0xffffffffu, se, off);
    if (i < a.Nq) {
      const size_t row = static_cast<size_t>(bh) * a.Nq + i;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx * 4 + c;
        if (j < a.Nb) scores[row * a.Nb + j] = sv[c];
      }
      if (tx == 0) {
        pm[row * a.n_ct + blockIdx.x] = mx;
        ps[row * a.n_ct + blockIdx.x] = se;
      }
    }
  }
}

// Key block j of routed row (query block i) is forced: a sink block, or one
// of the qr key blocks inside the query block (its diagonal).
__device__ __forceinline__ bool forced_block(const RouteArgs& a, int i, int j) {
  return j < a.n_sink || static_cast<unsigned>(j - i * a.qr) < static_cast<unsigned>(a.qr);
}

// The routed row (query block) whose list CSR row r (a 64-token block) holds.
__device__ __forceinline__ int64_t routed_row(const RouteArgs& a, int64_t r) {
  if (a.qr == 1) return r;
  const int64_t bh = r / a.Nb;
  return bh * a.Nq + (r - bh * a.Nb) / a.qr;
}

// -------------------------------------------------------------- select ---
// one warp per routed row (b, h, query block i); 8 rows per 256-thread CTA.
__global__ void __launch_bounds__(256) select_kernel(RouteArgs a) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= a.L.qrows) return;
  const int bh = static_cast<int>(row / a.Nq);
  const int i = static_cast<int>(row % a.Nq);
  uint32_t* bits = ws_ptr<uint32_t>(a.ws, a.L.bits) + row * a.words;
  int cnt = 0;
  bool flag = false;

  // rows that keep every key block: tau = 0 (outside top-mass), or a query
  // block meeting the prefix when prefix query rows are dense
  const bool row_all = a.keep_all || (a.mode == SA_ROUTE_DENSE_PREFIX_QUERIES && i < a.n_prefix_q);
  if (row_all) {
    for (int w = 0; w < a.words; ++w) {
      const int j = w * 32 + lane;
      const uint32_t m = __ballot_sync(full, j < a.Nb);
      if (lane == 0) bits[w] = m;
      cnt += __popc(m);
    }
  } else {
    const float* pm = ws_ptr<float>(a.ws, a.L.part_m) + row * a.n_ct;
    const float* ps = ws_ptr<float>(a.ws, a.L.part_s) + row * a.n_ct;
    float M = -INFINITY;
    for (int c = lane; c < a.n_ct; c += 32) M = fmaxf(M, pm[c]);
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(full, M, off));
    float Z = 0.f;
    for (int c = lane; c < a.n_ct; c += 32) Z += ps[c] * expf(pm[c] - M);
    for (int off = 16; off >= 1; off >>= 1) Z += __shfl_xor_sync(full, Z, off);
    const float T = M + logf(Z) + a.log_tau_over_nb;
    const float qn = ws_ptr<float>(a.ws, a.L.qnorm)[row];
    const float kmx = __int_as_float(ws_ptr<int>(a.ws, a.L.kmax)[bh]);
    const float* kn = ws_ptr<float>(a.ws, a.L.knorm) + static_cast<size_t>(bh) * a.Nb;
    const float gq = a.gamma * a.scale * qn;
    // T carries the worst logit error (the max over k of the bound above)
    // plus the roundings of the log-sum-exp itself: expf (2 ulp) and the
    // short shuffle-tree sums (relative 1e-6 of Z, so 1e-6 absolute in log Z),
    // logf (1 ulp of |log Z| <= 8) and three additions (ulps of |T|).
    const float err_row = gq * kmx + 2e-6f + 5e-7f * fabsf(T);
    float* srow = ws_ptr<float>(a.ws, a.L.scores) + row * a.Nb;
    if (a.mode == SA_ROUTE_TOP_MASS) {
      // p_j in place of the logits (this kernel is their last reader), then
      // a bisection on the cut: f(x) = sum of the p_j above x is decreasing;
      // keep the p_j above lo, where f(lo) >= tau > f(hi) and hi - lo is
      // below the spacing of distinct p. Rows whose fp32 masses at the cut,
      // or whose p on either side of the cut, are within the error bound of
      // tau or of each other go to the fp64 recheck.
      const float lse = M + logf(Z);
      for (int j = lane; j < a.Nb; j += 32) srow[j] = expf(srow[j] - lse);
      __syncwarp();
      auto mass_above = [&](float x) {
        float f = 0.f;
        for (int j = lane; j < a.Nb; j += 32) {
          const float pj = srow[j];
          f += pj > x ? pj : 0.f;
        }
        for (int off = 16; off >= 1; off >>= 1) f += __shfl_xor_sync(full, f, off);
        return f;
      };
      // the logit error bound becomes a relative error of each p (twice:
      // the logit and the log-sum-exp), plus the fp32 sums of up to Nb terms
      const float bound = 4.f * (gq * kmx + err_row) + (a.Nb / 32 + 8) * 2.4e-7f;
      float lo = 0.f, hi = 1.f, flo = 0.f, fhi = 0.f;
      bool take_all = false, take_none = false;
      if (a.tau <= 0.f) {
        take_none = true;
      } else {
        flo = mass_above(0.f);
        if (flo < a.tau) {
          take_all = true;            // even every block falls short of tau
          if (a.tau - flo <= bound) flag = true;
        } else {
          for (int itb = 0; itb < 40; ++itb) {
            const float mid = 0.5f * (lo + hi);
            const float fm = mass_above(mid);
            if (fm >= a.tau) { lo = mid; flo = fm; }
            else { hi = mid; fhi = fm; }
          }
          float p_last = INFINITY, p_next = 0.f;   // smallest kept, largest dropped
          for (int j = lane; j < a.Nb; j += 32) {
            const float pj = srow[j];
            if (pj > lo) p_last = fminf(p_last, pj);
            else p_next = fmaxf(p_next, pj);
          }
          for (int off = 16; off >= 1; off >>= 1) {
            p_last = fminf(p_last, __shfl_xor_sync(full, p_last, off));
            p_next = fmaxf(p_next, __shfl_xor_sync(full, p_next, off));
          }
          // masses: absolute error <= bound; order across the cut: each p carries a
          // relative error of about twice the logit bound, so a relative gap
          // below twice that may be an inversion
          const float rel = 4.f * (gq * kmx + err_row) + 4e-7f;
          if (flo - a.tau <= bound || a.tau - fhi <= bound || p_last - p_next <= rel * p_last)
            flag = true;
        }
      }
      for (int w = 0; w < a.words; ++w) {
        const int j = w * 32 + lane;
        bool keep = false;
        if (j < a.Nb) {
          const bool forced = forced_block(a, i, j);
          keep = forced || take_all || (!take_none && srow[j] > lo);
        }
        const uint32_t m = __ballot_sync(full, keep);
        if (lane == 0) bits[w] = m;
        cnt += __popc(m);
      }
    } else {
#pragma unroll 4
    for (int w = 0; w < a.words; ++w) {
      const int j = w * 32 + lane;
      bool keep = false;
      if (j < a.Nb) {
        const bool forced = forced_block(a, i, j);
        const float margin = srow[j] - T;
        keep = forced || (margin >= 0.f);
        if (!forced && fabsf(margin) <= fmaf(gq, kn[j], err_row)) flag = true;
      }
      const uint32_t m = __ballot_sync(full, keep);
      if (lane == 0) bits[w] = m;
      cnt += __popc(m);
    }
    }
  }
  flag = __any_sync(full, flag);
  if (lane == 0) {
    ws_ptr<int>(a.ws, a.L.counts)[row] = cnt;
    if (flag) {
      const int slot = atomicAdd(ws_ptr<int>(a.ws, a.L.nflag), 1);
      ws_ptr<int>(a.ws, a.L.flags)[slot] = static_cast<int>(row);
    }
  }
}

// ------------------------------------------------------------- recheck ---
// grid-stride over the queued rows; 256 threads (eight warps keep enough
// independent fp64 FMA chains in flight to cover the unit's latency); fp64
// throughout.
constexpr int kRecheckThreads = 256, kRecheckWarps = kRecheckThreads / 32;
static_assert(kRecheckWarps == 8, "the warp reductions below add eight partials");

__device__ __forceinline__ double sum8(const double* v) {
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

template <int D>
__global__ void __launch_bounds__(kRecheckThreads) recheck_kernel(RouteArgs a) {
  extern __shared__ __align__(16) double rs[];  // [D] qbar64 row, then [Nb] logits
  __shared__ double red[kRecheckWarps];
  __shared__ int redc[kRecheckWarps];
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double* qrow = rs;
  double* s64 = rs + D;
  const int nflag = *ws_ptr<int>(a.ws, a.L.nflag);
  const double* kb64 = ws_ptr<double>(a.ws, a.L.kbar64);
  const double* qb64 = ws_ptr<double>(a.ws, a.L.qbar64);

  for (int f = blockIdx.x; f < nflag; f += gridDim.x) {
    const int64_t row = ws_ptr<int>(a.ws, a.L.flags)[f];
    const int bh = static_cast<int>(row / a.Nq);
    const int i = static_cast<int>(row % a.Nq);
    for (int d = threadIdx.x; d < D; d += kRecheckThreads) qrow[d] = qb64[row * D + d];
    __syncthreads();
    // one key block per thread: the fp64 unit's throughput, not shuffle
    // latency, bounds this loop (four partial sums shorten the chains)
    for (int k = threadIdx.x; k < a.Nb; k += kRecheckThreads) {
      const double2* kr = reinterpret_cast<const double2*>(kb64 + (static_cast<size_t>(bh) * a.Nb + k) * D);
      double acc[4] = {0.0, 0.0, 0.0, 0.0};
#pragma unroll 8
      for (int d2 = 0; d2 < D / 2; d2 += 2) {
        const double2 x0 = kr[d2], x1 = kr[d2 + 1];
        acc[0] = fma(qrow[2 * d2], x0.x, acc[0]);
        acc[1] = fma(qrow[2 * d2 + 1], x0.y, acc[1]);
        acc[2] = fma(qrow[2 * d2 + 2], x1.x, acc[2]);
        acc[3] = fma(qrow[2 * d2 + 3], x1.y, acc[3]);
      }
      s64[k] = a.scale64 * ((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    __syncthreads();
    double m = -INFINITY;
    for (int k = threadIdx.x; k < a.Nb; k += kRecheckThreads) m = fmax(m, s64[k]);
    for (int off = 16; off >= 1; off >>= 1) m = fmax(m, __shfl_xor_sync(full, m, off));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
    for (int w = 1; w < kRecheckWarps; ++w) m = fmax(m, red[w]);
    __syncthreads();
    double z = 0.0;
    for (int k = threadIdx.x; k < a.Nb; k += kRecheckThreads) z += exp(s64[k] - m);
    for (int off = 16; off >= 1; off >>= 1) z += __shfl_xor_sync(full, z, off);
    if (lane == 0) red[warp] = z;
    __syncthreads();
    z = sum8(red);
    __syncthreads();
    // top-mass: the same bisection as the select kernel, in fp64 on the fp64
    // softmax (blocks above lo are kept, f(lo) >= tau > f(hi))
    double lo = 0.0;
    bool take_all = false, take_none = false;
    if (a.mode == SA_ROUTE_TOP_MASS) {
      for (int k = threadIdx.x; k < a.Nb; k += kRecheckThreads) s64[k] = exp(s64[k] - m) / z;
      __syncthreads();
      // one warp bisects (shuffle sums only); the others wait at the barrier
      if (warp == 0) {
        auto mass_above = [&](double x) {
          double f = 0.0;
          for (int k = lane; k < a.Nb; k += 32) f += s64[k] > x ? s64[k] : 0.0;
          for (int off = 16; off >= 1; off >>= 1) f += __shfl_xor_sync(full, f, off);
          return f;
        };
        int state = 0;                          // 0: cut at lo, 1: keep all, 2: keep none
        if (a.tau64 <= 0.0) {
          state = 2;
        } else if (mass_above(0.0) < a.tau64) {
          state = 1;
        } else {
          double hi = 1.0;
          for (int itb = 0; itb < 64; ++itb) {
            const double mid = 0.5 * (lo + hi);
            if (mass_above(mid) >= a.tau64) lo = mid;
            else hi = mid;
          }
        }
        if (lane == 0) {
          red[0] = lo;
          redc[0] = state;
        }
      }
      __syncthreads();
      lo = red[0];
      take_all = redc[0] == 1;
      take_none = redc[0] == 2;
      __syncthreads();
    }
    uint32_t* bits = ws_ptr<uint32_t>(a.ws, a.L.bits) + row * a.words;
    int cnt = 0;
    for (int w = warp; w < a.words; w += kRecheckWarps) {
      const int j = w * 32 + lane;
      bool keep = false;
      if (j < a.Nb) {
        const bool forced = forced_block(a, i, j);
        if (a.mode == SA_ROUTE_TOP_MASS)
          keep = forced || take_all || (!take_none && s64[j] > lo);
        else
          keep = forced || (exp(s64[j] - m) / z >= a.tau_over_nb);
      }
      const uint32_t bm = __ballot_sync(full, keep);
      if (lane == 0) bits[w] = bm;
      cnt += __popc(bm);
    }
    if (lane == 0) redc[warp] = cnt;
    __syncthreads();
    if (threadIdx.x == 0)
      ws_ptr<int>(a.ws, a.L.counts)[row] = redc[0] + redc[1] + redc[2] + redc[3] + redc[4] +
                                           redc[5] + redc[6] + redc[7];
    __syncthreads();
  }
}

// ---------------------------------------------------------------- scan ---
// one CTA of 1024 threads: row_ptr = exclusive scan of the counts of the
// CSR rows (each the count of its routed row).
__global__ void __launch_bounds__(1024) scan_kernel(RouteArgs a) {
  // one CTA; the rows are taken 1024 at a time (one count per thread, so the
  // loads and stores are coalesced), each pass scanned across the CTA and
  // offset by the running total of the passes before it
  __shared__ int64_t wsum[32];
  const int64_t n = a.L.rows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int* counts = ws_ptr<int>(a.ws, a.L.counts);
  int64_t carry = 0;
  // each pass loads the next pass's count before scanning its own, so the
  // global-load latency overlaps the scan
  int64_t c_next = tid < n ? counts[routed_row(a, tid)] : 0;
  for (int64_t r0 = 0; r0 < n; r0 += 1024) {
    const int64_t r = r0 + tid;
    const int64_t c = c_next;
    c_next = r + 1024 < n ? counts[routed_row(a, r + 1024)] : 0;
    int64_t incl = c;
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int64_t v = wsum[lane];
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      wsum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    if (r < n) a.row_ptr[r] = static_cast<int32_t>(carry + incl - c + (warp > 0 ? wsum[warp - 1] : 0));
    carry += wsum[31];
    __syncthreads();   // wsum is rewritten by the next pass
  }
  if (tid == 0) a.row_ptr[n] = static_cast<int32_t>(carry);
}

// ---------------------------------------------------------------- emit ---
// one warp per CSR row: set bits of its routed row's mask -> ascending key
// blocks.
__global__ void __launch_bounds__(256) emit_kernel(RouteArgs a) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= a.L.rows) return;
  const uint32_t* bits = ws_ptr<uint32_t>(a.ws, a.L.bits) + routed_row(a, row) * a.words;
  int64_t base = a.row_ptr[row];
  bool overflow = false;
  for (int w0 = 0; w0 < a.words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t u = (w < a.words) ? bits[w] : 0u;
    const int c = __popc(u);
    int incl = c;
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(full, incl, off);
      if (lane >= off) incl += v;
    }
    int64_t pos = base + (incl - c);
    while (u) {
      const int bpos = __ffs(u) - 1;
      if (pos < a.col_cap) a.col_idx[pos] = w * 32 + bpos;
      else overflow = true;
      ++pos;
      u &= u - 1;
    }
    base += __shfl_sync(full, incl, 31);
  }
  if (__any_sync(full, overflow) && lane == 0 && a.dev_status)
    atomicOr(a.dev_status, SA_DEV_CAPACITY);
}

// The router after pooling: logits, selection, recheck, CSR.
template <int D>
cudaError_t launch_select_d(const RouteArgs& a, cudaStream_t st) {
  const RouteLayout& L = a.L;
  cudaError_t e = cudaMemsetAsync(a.ws + L.nflag, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  {
    dim3 grid(a.n_ct, L.n_qt, a.B * a.H);
    score_kernel<D><<<grid, 256, 0, st>>>(a);
  }
  select_kernel<<<static_cast<unsigned>((L.qrows + 7) / 8), 256, 0, st>>>(a);
  {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = sizeof(double) * (D + a.Nb);
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(recheck_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    // top-mass: two queued rows per SM at a time (a row spends part of its
    // time in one warp's bisection, which the other row's warps overlap);
    // otherwise one, so that a row's dot products have the fp64 unit alone
    const int per_sm = a.mode == SA_ROUTE_TOP_MASS ? 2 : 1;
    recheck_kernel<D><<<per_sm * sms, kRecheckThreads, smem, st>>>(a);
  }
  scan_kernel<<<1, 1024, 0, st>>>(a);
  emit_kernel<<<static_cast<unsigned>((L.rows + 7) / 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

// Pooling (pa == nullptr: pool_kernel reads q, k) or the fused prologue.
template <int D>
cudaError_t launch_pool_d(const RouteArgs& a, const PrologueArgs* pa, cudaStream_t st) {
  const cudaError_t e =
      cudaMemsetAsync(a.ws + a.L.kmax, 0, sizeof(int) * static_cast<size_t>(a.B) * a.H, st);
  if (e != cudaSuccess) return e;
  dim3 grid(a.Nb, (a.H * D + 1023) / 1024, 2 * a.B);
  if (pa)
    prologue_kernel<D><<<grid, 128, 0, st>>>(a, *pa);
  else
    pool_kernel<D><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}
}  // namespace

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

RouteLayout route_layout(const sa_params& p) {
  RouteLayout L{};
  const int qblk = q_block_of(p);
  L.Nb = num_blocks(p.S);
  L.Nq = (p.S + qblk - 1) / qblk;
  L.n_ct = (L.Nb + kScoreTile - 1) / kScoreTile;
  L.n_qt = (L.Nq + kScoreTile - 1) / kScoreTile;
  L.words = (L.Nb + 31) / 32;
  const size_t bh = static_cast<size_t>(p.B) * p.H;
  L.rows = static_cast<int64_t>(bh) * L.Nb;
  L.qrows = static_cast<int64_t>(bh) * L.Nq;
  const size_t rows = static_cast<size_t>(L.rows);    // key blocks
  const size_t qrows = static_cast<size_t>(L.qrows);  // query blocks = routed rows
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align256(off + bytes); return o; };
  L.qbar32 = take(qrows * p.D * sizeof(float));
  L.kbar32 = take(rows * p.D * sizeof(float));
  L.qbar64 = take(qrows * p.D * sizeof(double));
  L.kbar64 = take(rows * p.D * sizeof(double));
  L.qnorm = take(qrows * sizeof(float));
  L.knorm = take(rows * sizeof(float));
  L.kmax = take(bh * sizeof(int));
  L.part_m = take(qrows * L.n_ct * sizeof(float));
  L.part_s = take(qrows * L.n_ct * sizeof(float));
  L.scores = take(qrows * static_cast<size_t>(L.Nb) * sizeof(float));
  L.bits = take(qrows * L.words * sizeof(uint32_t));
  L.counts = take(qrows * sizeof(int));
  L.nflag = take(sizeof(int));
  L.flags = take(qrows * sizeof(int));
  L.total = off;
  return L;
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t st) {
  const cudaError_t e = launch_pool(a, nullptr, st);
  return e == cudaSuccess ? launch_route_select(a, st) : e;
}

cudaError_t launch_pool(const RouteArgs& a, const PrologueArgs* pa, cudaStream_t st) {
  return a.D == 128 ? launch_pool_d<128>(a, pa, st) : launch_pool_d<64>(a, pa, st);
}

cudaError_t launch_route_select(const RouteArgs& a, cudaStream_t st) {
  return a.D == 128 ? launch_select_d<128>(a, st) : launch_select_d<64>(a, st);
}

}  // namespace sa
