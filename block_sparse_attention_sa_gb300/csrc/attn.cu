// attn.cu -- block-sparse flash-attention forward on sm_103a (tcgen05/TMEM/TMA).
//
// What is computed: for every query token of 64-token block i, exact softmax
// attention over the valid tokens of the key blocks routed to (b, h, i)
// (MiniAcc blog, "What is Sol attention?": only the selected pairs are
// computed; "MiniMax H3 runs on single 4090 with 4.44x speedup over dense
// execution", third paragraph: the exact prefix sink and the diagonal are
// part of every route). Dense mode lists every key block.
//
// Tiles. A tile is a 128-row query tile = query blocks 2p and 2p+1 of one
// head (tcgen05 M = 128; the route is per 64-row block). Its key walk is the
// union of the two blocks' key lists, two 64-key blocks per step (N = 128);
// a key block listed for only one of the two query blocks is masked to -inf
// for the other half's rows, so each row still sees exactly its own key set.
// The walk starts at the tile's diagonal block, where row maxima usually are.
//
// Persistent CTAs. One CTA per SM takes tiles from a global counter in
// (batch, head, pair) order, so concurrently running tiles share a head's
// K/V in L2. While one tile runs, a planner warp builds the next tile's key
// walk into the other half of a double buffer, the producer loads the next
// Q as soon as the last QK of the tile has read the old one, and the MMA
// warp queues the next tile's QKs during the current tile's epilogue.
//
// Split-K ping-pong. A tile's steps alternate between two softmax
// warpgroups: group 0 takes the even steps, group 1 the odd ones. Each group
// has its own S buffer, running max and sum, and O accumulator in TMEM
// (S0 S1 O0 O1 = 4 x 128 columns), so one group's softmax runs while the
// tensor pipe works on the other group's QK^T and PV. The two partial
// results are merged once per tile (rescaled to the common max, summed,
// divided by the common sum).
//
// Warps: 0-3 softmax group 0, 4-7 softmax group 1 (one thread per row =
// TMEM lane), 8 producer (lane 0: Q and K, lane 1: V), 9 MMA (converged;
// elect.sync issues), 10 planner, 11 idle. Step j: K(j) -> S[j%2] = Q K^T
// (bf16 x bf16 -> fp32) -> softmax(j) reads S, writes P (fp16) over the same
// columns -> O[j%2] += P V (fp16, A from TMEM) -> QK^T(j+2) reuses S[j%2].
// No data-dependent load sits inside a pipelined loop: the walk is built
// ahead by the planner. Every wait is bounded (SA_DEV_TIMEOUT) and an
// aborted CTA drains its own copies and MMAs and frees TMEM before it exits.
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sa_internal.cuh"

namespace sa {

namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // key rows per step (two key blocks)
constexpr int KST = 3;    // K stages
constexpr int VST = 2;    // V stages
constexpr int kThreads = 384;   // three warpgroups: softmax 0, softmax 1, control
constexpr int kGroupThreads = 128;
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kPlannerWarp = 10;  // warp 11: barriers only
// Register split (setmaxnreg). At launch ptxas gives every thread
// kLaunchRegs (65536 / 384 rounded down to a multiple of 8); the two softmax
// warpgroups then grow to kSoftmaxRegs and the control warpgroup shrinks
// to kControlRegs: 2*128*216 + 128*64 = 63,488 <= 384*168 = 64,512, and per
// SM sub-partition (one warp of each warpgroup) 216 + 216 + 64 <= 512.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 216;
constexpr int kControlRegs = 64;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;
constexpr int kColS = 0;      // S[g] at columns [128 g, 128 g + 128)
constexpr int kColO = 256;    // O[g] at columns [256 + 128 g, 256 + 128 g + D)
// Lazy rescale: the running max moves only when a block max exceeds it by
// more than 2^14, so P <= 16384 stays well inside fp16; values that fall
// below fp16's normal range weigh under 2^-28 of the row max.
constexpr float kRescaleLog2 = 14.0f;

template <int D>
struct Smem {
  static constexpr int kRegion = BM * 128;            // one 64-wide K slice of 128 rows
  static constexpr int kQ = 0;
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kKBytes = BN * D * 2;
  static constexpr int kV = kK + KST * kKBytes;
  static constexpr int kVBytes = BN * D * 2;
  static constexpr int kVHalf = D * 128;              // one 64-key half of a V^T stage
  static constexpr int kBar = kV + VST * kVBytes;
  // barriers (counts in the init loop below)
  static constexpr int bInfoFull = 0;                 // [2] planner wrote walk x
  static constexpr int bInfoEmpty = bInfoFull + 2;    // [2] every consumer is done with walk x
  static constexpr int bQFull = bInfoEmpty + 2;       // Q of the current tile landed
  static constexpr int bQEmpty = bQFull + 1;          // the tile's last QK is done with Q
  static constexpr int bKFull = bQEmpty + 1;          // [KST]
  static constexpr int bKEmpty = bKFull + KST;        // [KST]
  static constexpr int bVFull = bKEmpty + KST;        // [VST]
  static constexpr int bVEmpty = bVFull + VST;        // [VST]
  static constexpr int bSFull = bVEmpty + VST;        // [2] QK of group g's step done
  static constexpr int bPFull = bSFull + 2;           // [2] softmax of group g's step done
  static constexpr int bTileDone = bPFull + 2;        // every PV of the tile done
  static constexpr int bXch = bTileDone + 1;          // [2] both groups posted (m, l)
  static constexpr int bOFree = bXch + 2;             // both groups have read O
  static constexpr int bFin = bOFree + 1;             // every MMA done (exit)
  static constexpr int kNumBars = bFin + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kHdr = kMisc + 16;             // [2][4] walk headers: b, h, pair, n
  static constexpr int kXch = kHdr + 32;              // [2 parity][2 groups][2 (m, l)][128]
  static constexpr int kBits = kXch + 2 * 2 * 2 * BM * 4;
  static constexpr int kInfo = kBits + 2 * (kMaxNbAttn / 32) * 4;  // [2][kMaxNbAttn] walks
  static constexpr int kEnd = kInfo + 2 * kMaxNbAttn * 2;
  static constexpr int kBytes = kEnd + 1024;          // slack to align the base to 1 KB
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void set_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

// Wait sites, recorded as bit (8 + site) next to SA_DEV_TIMEOUT when a wait
// gives up, so a status word names the stage that stalled.
enum WaitSite {
  kSiteKStage = 0, kSiteVStage, kSiteQFull, kSiteKFull, kSitePFull, kSiteVFull,
  kSiteSFull, kSiteFin, kSiteInfo, kSiteOFree
};

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void note_timeout(int32_t* st, int site) {
  set_status(st, SA_DEV_TIMEOUT | (1 << (8 + site)));
}

// max over 64 fp32 values (bit patterns): eight chains of three-input max.
__device__ __forceinline__ float max64(const uint32_t* v) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(__uint_as_float(v[i]), __uint_as_float(v[8 + i]));
#pragma unroll
  for (int i = 16; i < 64; i += 16)
#pragma unroll
    for (int c = 0; c < 8; ++c)
      m[c] = fmax3(m[c], __uint_as_float(v[i + c]), __uint_as_float(v[i + 8 + c]));
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(fmax3(m[3], m[4], m[5]), m[6], m[7]));
}

// p = 2^(s * c - m) for 64 logits, packed as fp16 pairs into 32 words;
// returns the fp32 sum of the p. The scale-and-subtract and the running sums
// use paired fp32 arithmetic (four independent sum chains).
__device__ __forceinline__ float exp_pack64(const uint32_t* v, float c, float negm,
                                            uint32_t* pk) {
  const uint64_t c2 = f2_pack(c, c), m2 = f2_pack(negm, negm);
  uint64_t acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0ull;
#pragma unroll
  for (int u = 0; u < 64; u += 2) {
    const uint64_t y = f2_fma(f2_pack(__uint_as_float(v[u]), __uint_as_float(v[u + 1])), c2, m2);
    float y0, y1;
    f2_unpack(y, y0, y1);
    const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
    acc[(u >> 1) & 3] = f2_add(acc[(u >> 1) & 3], f2_pack(p0, p1));
    pk[u >> 1] = pack_half2(p0, p1);
  }
  const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float lo, hi;
  f2_unpack(t, lo, hi);
  return lo + hi;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_vt, const AttnArgs a) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nb = a.Nb, S = a.S;
  const unsigned full = 0xffffffffu;

  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const AbortSignal abort_sig{abort_flag, a.dev_status};
  const volatile int never_flag = 0;
  const AbortSignal drain_sig{&never_flag, nullptr};  // drains wait out their own limit
  volatile int* hdr = reinterpret_cast<volatile int*>(smem + L::kHdr);
  uint16_t* info = reinterpret_cast<uint16_t*>(smem + L::kInfo);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  auto fail = [&](int site) {
    *abort_flag = 1;
    note_timeout(a.dev_status, site);
  };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    // Arrival counts. No barrier can complete its next phase before each of
    // its waiters has seen the current one, so parity waits never fall a
    // full round behind: every next phase needs work the waiter releases
    // after its wait (the walk buffers need all their consumers; QK(j+2)
    // follows p_full(j); a stage is refilled only after it was freed; the
    // next tile's first PV waits for o_free, which needs every softmax
    // thread past its tile_done wait; and so on).
    for (int i = 0; i < L::kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == L::bInfoEmpty || i == L::bInfoEmpty + 1) cnt = 3 + kSoftmaxThreads;
      if (i == L::bPFull || i == L::bPFull + 1) cnt = kGroupThreads;
      if (i == L::bXch || i == L::bXch + 1 || i == L::bOFree) cnt = kSoftmaxThreads;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // Each role branch resizes its registers first thing and does not rejoin
  // the others before the final barrier, so ptxas can give each branch its
  // own budget.
  if (warp == kPlannerWarp) {
    regs_dec<kControlRegs>();
    // -------------------------------------------------------------- planner
    // Takes tiles in order from the global counter and writes each tile's
    // key walk (the rotated union of its two query blocks' key lists, with
    // a 2-bit membership mask per key block) into walk buffer it % 2.
    uint32_t* bmA = reinterpret_cast<uint32_t*>(smem + L::kBits);
    uint32_t* bmB = bmA + kMaxNbAttn / 32;
    for (int it = 0;; ++it) {
      const int x = it & 1;
      int tile = 0;
      if (lane == 0) tile = atomicAdd(a.tile_counter, 1);
      tile = __shfl_sync(full, tile, 0);
      if (*abort_flag) tile = a.n_tiles;
      if (it >= 2 && !mbar_wait_warp(bar(L::bInfoEmpty + x), ((it >> 1) - 1) & 1, abort_sig)) {
        if (lane == 0) fail(kSiteInfo);
        break;
      }
      volatile int* hd = hdr + 4 * x;
      uint16_t* inf = info + x * kMaxNbAttn;
      if (tile >= a.n_tiles) {
        if (lane == 0) hd[3] = -1;   // no more tiles: every role leaves its loop
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bInfoFull + x));
        break;
      }
      const int pair = tile % a.n_pairs;
      const int bh = tile / a.n_pairs;
      const int h = bh % a.H, b = bh / a.H;
      const int qb0 = 2 * pair;
      const bool has_qb1 = qb0 + 1 < Nb;
      // Union of the two query blocks' key lists with a 2-bit membership mask
      // per key block (bit 0: block 2p lists it, bit 1: block 2p+1 does),
      // ascending but rotated to start at the tile's own diagonal block: the
      // row maxima usually sit near the diagonal, so taking it first keeps
      // later steps from raising the running max (each raise rescales O).
      const int words = (Nb + 31) >> 5;
      int bad = 0;
      if (a.row_ptr == nullptr) {
        const uint16_t m = has_qb1 ? 3 : 1;
        for (int j = lane; j < Nb; j += 32)
          inf[(j - qb0 + Nb) % Nb] = static_cast<uint16_t>((j << 2) | m);
        if (lane == 0) hd[3] = Nb;
      } else {
        for (int w = lane; w < words; w += 32) { bmA[w] = 0u; bmB[w] = 0u; }
        __syncwarp();
        for (int half = 0; half < 2; ++half) {
          if (half == 1 && !has_qb1) break;
          const int64_t r = (static_cast<int64_t>(b) * a.H + h) * Nb + qb0 + half;
          const int beg = a.row_ptr[r], end = a.row_ptr[r + 1];
          if (beg < 0 || end < beg || end - beg > Nb) { bad = 1; continue; }
          uint32_t* bm = half ? bmB : bmA;
          for (int e = beg + lane; e < end; e += 32) {
            const int j = a.col_idx[e];
            if (j < 0 || j >= Nb) bad = 1;
            else atomicOr(&bm[j >> 5], 1u << (j & 31));
          }
        }
        __syncwarp();
        // count the union and the entries below the diagonal (the rotation)
        int total = 0, below = 0;
        for (int w = lane; w < words; w += 32) {
          const uint32_t u = bmA[w] | bmB[w];
          total += __popc(u);
          const int lo = w * 32;
          const uint32_t below_mask =
              qb0 >= lo + 32 ? 0xffffffffu : (qb0 <= lo ? 0u : ((1u << (qb0 - lo)) - 1u));
          below += __popc(u & below_mask);
        }
        for (int off = 16; off >= 1; off >>= 1) {
          total += __shfl_xor_sync(0xffffffffu, total, off);
          below += __shfl_xor_sync(0xffffffffu, below, off);
        }
        int base = 0;
        for (int w0 = 0; w0 < words; w0 += 32) {
          const int w = w0 + lane;
          const uint32_t ua = w < words ? bmA[w] : 0u, ub = w < words ? bmB[w] : 0u;
          uint32_t u = ua | ub;
          const int c = __popc(u);
          int incl = c;
          for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
          }
          int pos = base + incl - c;
          while (u) {
            const int bit = __ffs(u) - 1;
            const uint32_t m = ((ua >> bit) & 1u) | (((ub >> bit) & 1u) << 1);
            int rp = pos - below;
            if (rp < 0) rp += total;
            inf[rp] = static_cast<uint16_t>(((w * 32 + bit) << 2) | m);
            ++pos;
            u &= u - 1;
          }
          base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) hd[3] = total;
      }
      if (__any_sync(full, bad) && lane == 0) set_status(a.dev_status, SA_DEV_BAD_ROUTE);
      if (lane == 0) {
        hd[0] = b;
        hd[1] = h;
        hd[2] = pair;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bInfoFull + x));
    }
  } else if (warp == kProducerWarp) {
    regs_dec<kControlRegs>();
    // ------------------------------------------------------------- producer
    // Lane 0 streams Q and K, lane 1 streams V, each as far ahead as its
    // ring allows. Each lane waits for all of its own copies to land before
    // it leaves, so no copy can outlive the CTA's shared memory.
    if (lane == 0) {
      int issued[KST] = {0};
      int q_loads = 0, kcnt = 0;
      for (int it = 0;; ++it) {
        const int x = it & 1;
        if (!mbar_wait(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) { fail(kSiteInfo); break; }
        const volatile int* hd = hdr + 4 * x;
        const int n = hd[3];
        if (n < 0) break;
        const int b = hd[0], h = hd[1], qb0 = 2 * hd[2];
        const uint16_t* inf = info + x * kMaxNbAttn;
        // the previous tile's QKs are done with the Q buffer
        if (it >= 1 && !mbar_wait(bar(L::bQEmpty), (it - 1) & 1, abort_sig)) { fail(kSiteQFull); break; }
        mbar_arrive_expect_tx(bar(L::bQFull), L::kQBytes);
        ++q_loads;
        for (int qh = 0; qh < 2; ++qh)
          for (int dh = 0; dh < D / 64; ++dh)
            tma_load_4d(sbase + L::kQ + dh * L::kRegion + qh * 8192, &tm_q, bar(L::bQFull),
                        dh * 64, (qb0 + qh) * kBlock, h, b);
        const int n_steps = (n + 1) >> 1;
        bool ok = true;
        for (int j = 0; j < n_steps; ++j, ++kcnt) {
          const int nblk = (2 * j + 1 < n) ? 2 : 1;
          const int ks = kcnt % KST;
          if (kcnt >= KST && !mbar_wait(bar(L::bKEmpty + ks), ((kcnt / KST) - 1) & 1, abort_sig)) {
            fail(kSiteKStage);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(L::bKFull + ks), nblk * kBlock * D * 2);
          ++issued[ks];
          for (int kh = 0; kh < nblk; ++kh) {
            const int jk = inf[2 * j + kh] >> 2;
            for (int dh = 0; dh < D / 64; ++dh)
              tma_load_4d(sbase + L::kK + ks * L::kKBytes + dh * L::kRegion + kh * 8192, &tm_k,
                          bar(L::bKFull + ks), dh * 64, jk * kBlock, h, b);
          }
        }
        if (!ok) break;
        mbar_arrive(bar(L::bInfoEmpty + x));
      }
      if (q_loads) mbar_wait(bar(L::bQFull), (q_loads - 1) & 1, drain_sig);
      for (int s2 = 0; s2 < KST; ++s2)
        if (issued[s2]) mbar_wait(bar(L::bKFull + s2), (issued[s2] - 1) & 1, drain_sig);
    } else if (lane == 1) {
      int issued[VST] = {0};
      int vcnt = 0;
      for (int it = 0;; ++it) {
        const int x = it & 1;
        if (!mbar_wait(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) { fail(kSiteInfo); break; }
        const volatile int* hd = hdr + 4 * x;
        const int n = hd[3];
        if (n < 0) break;
        const int bh = hd[0] * a.H + hd[1];
        const uint16_t* inf = info + x * kMaxNbAttn;
        const int n_steps = (n + 1) >> 1;
        bool ok = true;
        for (int j = 0; j < n_steps; ++j, ++vcnt) {
          const int nblk = (2 * j + 1 < n) ? 2 : 1;
          const int vs = vcnt % VST;
          if (vcnt >= VST && !mbar_wait(bar(L::bVEmpty + vs), ((vcnt / VST) - 1) & 1, abort_sig)) {
            fail(kSiteVStage);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(L::bVFull + vs), nblk * kBlock * D * 2);
          ++issued[vs];
          for (int kh = 0; kh < nblk; ++kh) {
            const int jk = inf[2 * j + kh] >> 2;
            tma_load_3d(sbase + L::kV + vs * L::kVBytes + kh * L::kVHalf, &tm_vt,
                        bar(L::bVFull + vs), jk * kBlock, 0, bh);
          }
        }
        if (!ok) break;
        mbar_arrive(bar(L::bInfoEmpty + x));
      }
      for (int s2 = 0; s2 < VST; ++s2)
        if (issued[s2]) mbar_wait(bar(L::bVFull + s2), (issued[s2] - 1) & 1, drain_sig);
    }
  } else if (warp == kMmaWarp) {
    regs_dec<kControlRegs>();
    // ------------------------------------------------------------------ MMA
    // The whole warp runs this loop in step (warp-uniform waits); elect.sync
    // picks the lane that issues each batch of MMAs and each commit.
    constexpr uint32_t kIdQK128 = idesc_f16(BM, 128, 1);
    constexpr uint32_t kIdQK64 = idesc_f16(BM, 64, 1);
    constexpr uint32_t kIdPV = idesc_f16(BM, D, 0);
    // Descriptors: Q's K slices (start address stepped by 32 bytes inside a
    // 128-byte swizzle row, then by one 16 KB region per 64 elements), and
    // the K/V stage bases.
    uint64_t qd[D / 16];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      qd[kk] = sdesc_kmajor_sw128(sbase + L::kQ + (kk >> 2) * L::kRegion + (kk & 3) * 32);
    const uint64_t k0 = sdesc_kmajor_sw128(sbase + L::kK);
    const uint64_t v0 = sdesc_kmajor_sw128(sbase + L::kV);
    int kcnt = 0, vcnt = 0;
    int grp_steps0 = 0, grp_steps1 = 0;  // steps of each group in earlier tiles
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int x = it & 1;
      if (!mbar_wait_warp(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) {
        if (lane == 0) fail(kSiteInfo);
        break;
      }
      const int n = hdr[4 * x + 3];
      if (n < 0) break;
      const int n_steps = (n + 1) >> 1;
      if (!mbar_wait_warp(bar(L::bQFull), it & 1, abort_sig)) {
        if (lane == 0) fail(kSiteQFull);
        break;
      }
      tc_fence_after();
      auto issue_qk = [&](int j) -> bool {
        const int ks = kcnt % KST;
        if (!mbar_wait_warp(bar(L::bKFull + ks), (kcnt / KST) & 1, abort_sig)) {
          if (lane == 0) fail(kSiteKFull);
          return false;
        }
        tc_fence_after();
        const uint32_t idesc = (2 * j + 1 < n) ? kIdQK128 : kIdQK64;
        const uint32_t d_tmem = tmem + kColS + (j & 1) * 128;
        const uint64_t kb = k0 + static_cast<uint64_t>(ks * (L::kKBytes >> 4));
        uint64_t kd[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          kd[kk] = kb + static_cast<uint64_t>(((kk >> 2) * L::kRegion + (kk & 3) * 32) >> 4);
#pragma unroll
        for (int g = 0; g < D / 64; ++g)
          umma_ss_x4_elect(d_tmem, qd[4 * g], qd[4 * g + 1], qd[4 * g + 2], qd[4 * g + 3],
                           kd[4 * g], kd[4 * g + 1], kd[4 * g + 2], kd[4 * g + 3], idesc, g > 0);
        umma_commit_elect(bar(L::bSFull + (j & 1)));
        umma_commit_elect(bar(L::bKEmpty + ks));
        if (j == n_steps - 1) umma_commit_elect(bar(L::bQEmpty));  // Q no longer read
        ++kcnt;
        return true;
      };
      if (n_steps == 0) umma_commit_elect(bar(L::bQEmpty));
      for (int j = 0; j < 2 && j < n_steps && ok; ++j) ok = issue_qk(j);
      if (!ok) break;
      // the previous tile's epilogue has read both O accumulators
      if (it >= 1 && !mbar_wait_warp(bar(L::bOFree), (it - 1) & 1, abort_sig)) {
        if (lane == 0) fail(kSiteOFree);
        break;
      }
      tc_fence_after();
      for (int j = 0; j < n_steps && ok; ++j) {
        const int g = j & 1;
        const int gstep = (g == 0 ? grp_steps0 : grp_steps1) + (j >> 1);
        if (!mbar_wait_warp(bar(L::bPFull + g), gstep & 1, abort_sig)) {
          if (lane == 0) fail(kSitePFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const int vs = vcnt % VST;
        if (!mbar_wait_warp(bar(L::bVFull + vs), (vcnt / VST) & 1, abort_sig)) {
          if (lane == 0) fail(kSiteVFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = tmem + kColS + g * 128;   // P(j) over S(j)
        const uint32_t od = tmem + kColO + g * 128;   // this group's O
        const uint64_t vb = v0 + static_cast<uint64_t>(vs * (L::kVBytes >> 4));
        umma_ts_x4_elect(od, pa, vb, vb + 2, vb + 4, vb + 6, kIdPV, j >= 2);
        if (2 * j + 1 < n) {
          const uint64_t vh = vb + (L::kVHalf >> 4);
          umma_ts_x4_elect(od, pa + 32, vh, vh + 2, vh + 4, vh + 6, kIdPV, 1u);
        }
        umma_commit_elect(bar(L::bVEmpty + vs));
        ++vcnt;
        // S[g] now belongs to QK(j+2): PV(j), the last reader of P(j), was
        // issued just before, and the tensor pipe runs the MMAs in order.
        if (j + 2 < n_steps && !issue_qk(j + 2)) ok = false;
      }
      grp_steps0 += (n_steps + 1) >> 1;
      grp_steps1 += n_steps >> 1;
      if (!ok) break;
      umma_commit_elect(bar(L::bTileDone));
      if (elect_one()) mbar_arrive(bar(L::bInfoEmpty + x));
    }
    // Every MMA issued above completes before TMEM is released.
    umma_commit_elect(bar(L::bFin));
    mbar_wait_warp(bar(L::bFin), 0, drain_sig);
  } else if (warp > kPlannerWarp) {
    regs_dec<kControlRegs>();   // warp 11: nothing to do but the barriers
  } else {
    regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------- softmax
    const int grp = warp >> 2;                 // 0: even steps, 1: odd steps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;         // tile row == TMEM lane
    const int qh = r >> 6;                     // query block of this row (warp-uniform)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = kColS + grp * 128;
    const uint32_t o_col = kColO + grp * 128;
    const int last_valid = S - (Nb - 1) * kBlock;  // tokens in the last block
    const float cl2 = a.scale_log2;
    float* xch = reinterpret_cast<float*>(smem + L::kXch);
    int gstep = 0;                             // this group's steps so far (all tiles)
    bool ok = true;

    for (int it = 0; ok; ++it) {
      const int x = it & 1;
      if (!mbar_wait_warp(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) {
        if (lane == 0) fail(kSiteInfo);
        break;
      }
      const volatile int* hd = hdr + 4 * x;
      const int n = hd[3];
      if (n < 0) break;
      const int b = hd[0], h = hd[1], qb0 = 2 * hd[2];
      const uint16_t* inf = info + x * kMaxNbAttn;
      const int n_steps = (n + 1) >> 1;
      const int t = qb0 * kBlock + r;          // query token
      float m_run = -INFINITY, l_run = 0.f;

      for (int j = grp; j < n_steps; j += 2, ++gstep) {
        if (!mbar_wait_warp(bar(L::bSFull + grp), gstep & 1, abort_sig)) {
          if (lane == 0) fail(kSiteSFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const int nblk = (2 * j + 1 < n) ? 2 : 1;
        const uint32_t e0 = inf[2 * j];
        const uint32_t e1 = nblk == 2 ? inf[2 * j + 1] : 0u;
        const bool mem0 = (e0 >> qh) & 1u;
        const bool mem1 = nblk == 2 && ((e1 >> qh) & 1u);
        uint32_t sr[BN];
        if (mem0) {
          tmem_ld32(lane_base + s_col, sr);
          tmem_ld32(lane_base + s_col + 32, sr + 32);
        }
        if (mem1) {
          tmem_ld32(lane_base + s_col + 64, sr + 64);
          tmem_ld32(lane_base + s_col + 96, sr + 96);
        }
        tmem_wait_ld();
        // the ragged last block: keys past S weigh exactly zero
        if (mem0 && static_cast<int>(e0 >> 2) == Nb - 1) {
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u >= last_valid) sr[u] = __float_as_uint(-INFINITY);
        }
        if (mem1 && static_cast<int>(e1 >> 2) == Nb - 1) {
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u >= last_valid) sr[64 + u] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
        if (mem0) mx = fmaxf(mx, max64(sr));
        if (mem1) mx = fmaxf(mx, max64(sr + 64));
        const float bmax = mx * cl2;           // the scale is positive: max commutes
        float m_new = m_run;
        if (bmax > m_run + kRescaleLog2) m_new = bmax;  // also the first finite block
        const bool rescale = (m_new != m_run) && (m_run != -INFINITY);
        const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
        const float negm = -m_new;
        // P(j) over the consumed S(j) columns: keys 0-63 -> columns 0-31,
        // keys 64-127 -> columns 32-63 (two fp16 per column); each half is
        // stored as soon as it is ready.
        float rs = 0.f;
        {
          uint32_t pk[32];
          if (mem0) rs += exp_pack64(sr, cl2, negm, pk);
          else {
#pragma unroll
            for (int u = 0; u < 32; ++u) pk[u] = 0u;
          }
          tmem_st32(lane_base + s_col, pk);
        }
        if (nblk == 2) {
          uint32_t pk[32];
          if (mem1) rs += exp_pack64(sr + 64, cl2, negm, pk);
          else {
#pragma unroll
            for (int u = 0; u < 32; ++u) pk[u] = 0u;
          }
          tmem_st32(lane_base + s_col + 32, pk);
        }
        l_run = l_run * alpha + rs;
        m_run = m_new;
        if (__any_sync(0xffffffffu, rescale)) {
          // S(j) ready means QK(j) is done, and QK(j) was issued after this
          // group's previous PV(j-2): that PV is done too, and PV(j) waits for
          // p_full(j), so O[grp] is stable here without another wait.
  #pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + o_col + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(lane_base + o_col + 32 * c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::bPFull + grp));
      }
      if (!ok) break;
      mbar_arrive(bar(L::bInfoEmpty + x));     // done with this walk

      // -------------------------------------------------------- epilogue
      // Merge the two groups' partial results for this row: both threads of
      // the row (same lane, groups 0 and 1) post (m, l), then each writes
      // half of the output columns.
      float* xs = xch + x * (2 * 2 * BM);
      xs[(grp * 2 + 0) * BM + r] = m_run;
      xs[(grp * 2 + 1) * BM + r] = l_run;
      mbar_arrive(bar(L::bXch + x));
      if (!mbar_wait_warp(bar(L::bXch + x), (it >> 1) & 1, abort_sig) ||
          !mbar_wait_warp(bar(L::bTileDone), it & 1, abort_sig)) {
        if (lane == 0) fail(kSiteFin);
        ok = false;
        break;
      }
      tc_fence_after();
      const float m0 = xs[0 * BM + r], l0 = xs[1 * BM + r];
      const float m1 = xs[2 * BM + r], l1 = xs[3 * BM + r];
      const float m = fmaxf(m0, m1);
      const float s0 = l0 > 0.f ? fast_exp2(m0 - m) : 0.f;   // group 0's weight
      const float s1 = l1 > 0.f ? fast_exp2(m1 - m) : 0.f;   // group 1's weight
      const float l_tot = l0 * s0 + l1 * s1;
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float w0 = s0 * inv_l, w1 = s1 * inv_l;
      const bool row_ok = t < S;
      uint16_t* orow = a.o + b * a.os[0] + static_cast<int64_t>(t) * a.os[1] + h * a.os[2] +
                       grp * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t col = grp * (D / 2) + 32 * c;
        uint32_t oa[32], ob[32];
        tmem_ld32(lane_base + kColO + col, oa);
        tmem_ld32(lane_base + kColO + 128 + col, ob);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              // a group with no weight may not have written its O in this
              // tile: select, never multiply, so stale TMEM cannot leak in
              const float xa = s0 > 0.f ? __uint_as_float(oa[8 * v + u]) * w0 : 0.f;
              const float xb = s1 > 0.f ? __uint_as_float(ob[8 * v + u]) * w1 : 0.f;
              f[u] = xa + xb;
            }
            uint4 wv;
            wv.x = pack_bf162(f[0], f[1]);
            wv.y = pack_bf162(f[2], f[3]);
            wv.z = pack_bf162(f[4], f[5]);
            wv.w = pack_bf162(f[6], f[7]);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * v) = wv;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::bOFree));             // both O accumulators read
      if (row_ok && grp == 0 && a.lse) {
        const float lse = l_tot > 0.f ? m * 0.69314718055994531f + logf(l_tot) : -INFINITY;
        a.lse[(static_cast<int64_t>(b) * a.H + h) * S + t] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// V [B,S,H,D] bf16 -> vt [B*H][D][s_pad] fp16. grid (ceil(S/64), H, B), 256 threads.
template <int D>
__global__ void __launch_bounds__(256)
pack_v_kernel(const uint16_t* __restrict__ v, int64_t vs0, int64_t vs1, int64_t vs2, int S, int H,
              int s_pad, uint16_t* __restrict__ vt, int32_t* dev_status) {
  __shared__ uint16_t tile[kBlock][D + 8];
  const int s0 = blockIdx.x * kBlock, h = blockIdx.y, b = blockIdx.z;
  bool range = false;
  constexpr int VPR = D / 8;  // 16-byte vectors per token row
  for (int idx = threadIdx.x; idx < kBlock * VPR; idx += 256) {
    const int r = idx / VPR, c = (idx % VPR) * 8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (s0 + r < S)
      w = __ldg(reinterpret_cast<const uint4*>(v + b * vs0 + static_cast<int64_t>(s0 + r) * vs1 +
                                               h * vs2 + c));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float f = __uint_as_float((hh ? (ww[u] & 0xffff0000u) : (ww[u] << 16)));
        const __half hv = __float2half_rn(f);
        if (isinf(__half2float(hv)) && !isinf(f)) range = true;
        tile[r][c + 2 * u + hh] = *reinterpret_cast<const uint16_t*>(&hv);
      }
    }
  }
  __syncthreads();
  uint16_t* dst = vt + (static_cast<int64_t>(b) * H + h) * D * s_pad;
  for (int idx = threadIdx.x; idx < D * (kBlock / 8); idx += 256) {
    const int d = idx / (kBlock / 8), c = (idx % (kBlock / 8)) * 8;
    if (s0 + c >= s_pad) continue;
    uint16_t e[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e[u] = tile[c + u][d];
    uint4 w;
    w.x = e[0] | (static_cast<uint32_t>(e[1]) << 16);
    w.y = e[2] | (static_cast<uint32_t>(e[3]) << 16);
    w.z = e[4] | (static_cast<uint32_t>(e[5]) << 16);
    w.w = e[6] | (static_cast<uint32_t>(e[7]) << 16);
    *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(d) * s_pad + s0 + c) = w;
  }
  if (__syncthreads_or(range) && threadIdx.x == 0) set_status(dev_status, SA_DEV_RANGE);
}

template <int D>
cudaError_t launch_attn_d(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  constexpr int smem = Smem<D>::kBytes;
  static_assert(smem <= 227 * 1024, "attention tile does not fit shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.n_tiles < sms ? a.n_tiles : sms;   // persistent: one CTA per SM
  attn_fwd_kernel<D><<<grid, kThreads, smem, st>>>(m.q, m.k, m.vt, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_v(const uint16_t* v, const int64_t vs[3], int B, int S, int H, int D,
                          int s_pad, uint16_t* vt, int32_t* dev_status, cudaStream_t st) {
  dim3 grid((S + kBlock - 1) / kBlock, H, B);
  if (D == 128)
    pack_v_kernel<128><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], S, H, s_pad, vt, dev_status);
  else
    pack_v_kernel<64><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], S, H, s_pad, vt, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_attn(int D, const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  return D == 128 ? launch_attn_d<128>(m, a, st) : launch_attn_d<64>(m, a, st);
}

}  // namespace sa
