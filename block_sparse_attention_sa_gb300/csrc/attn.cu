// attn.cu -- block-sparse flash-attention forward on sm_103a (tcgen05/TMEM/TMA).
//
// What is computed: for every query token of 64-token block i, exact softmax
// attention over the valid tokens of the key blocks routed to (b, h, i)
// (MiniAcc blog, "What is Sol attention?": only the selected pairs are
// computed; "MiniMax H3 runs on single 4090 with 4.44x speedup over dense
// execution", third paragraph: the exact prefix sink and the diagonal are
// part of every route). Dense mode lists every key block.
//
// Tile and roles. One CTA owns a 128-row query tile = query blocks 2p and
// 2p+1 of one head (tcgen05 M = 128; the route is per 64-row block). It
// walks the ascending union of the two blocks' key lists, two 64-key blocks
// per step (N = 128); a key block listed for only one of the two query
// blocks is masked to -inf for the other half's rows, so each row still sees
// exactly its own key set. Ten warps:
//   warps 0-7  softmax + epilogue: two threads per query row (TMEM lane);
//              warps 0-3 take the step's first key block and the first half
//              of O's columns, warps 4-7 (same lanes) the second; the pair
//              swaps its row max through shared memory every step
//   warp  8    builds the tile's key-block union in shared memory, then one
//              lane issues every TMA load (Q once; K and V^T per step)
//   warp  9    allocates TMEM; one lane issues every tcgen05.mma
// Pipeline per step j: K(j) -> S[j%3] = Q K^T (bf16, fp32 in TMEM)
//   -> softmax(j) reads S, writes P (fp16) back over the same TMEM columns,
//   and rescales O in TMEM only when the running max moved by more than 2^8
//   -> O += P V with P read from TMEM (fp16, fp32 accumulation). With three
//   S buffers the MMA thread issues PV(j) as soon as P(j) is ready and then
//   QK(j+3), so QK(j+1) and QK(j+2) are already queued while softmax(j)
//   runs; softmax waits for the previous PV only when it has to rescale O.
// The producer alone reads the route, before the pipeline starts, so no
// data-dependent load sits inside the pipelined loops.
// Every wait is bounded (SA_DEV_TIMEOUT) and an aborted CTA drains its own
// copies and MMAs and frees TMEM before it exits.
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sa_internal.cuh"

namespace sa {

namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // key rows per step (two key blocks)
constexpr int KST = 3;    // K stages (= S buffers: s_full[j%3] also frees K stage j%3)
constexpr int VST = 2;    // V stages (= o_ready barriers: o_ready[j%2] frees V stage j%2)
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr int kNumS = 3;                 // S/P buffers in TMEM (128 columns each)
constexpr int kColO = kNumS * 128;       // O accumulator columns [384, 384 + D)
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold: P <= 2^8 in fp16

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
  // barriers
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bVFull = bKFull + KST;
  // QK(j) done (s_full[j%3]) frees K stage j%3, and PV(j) done
  // (o_ready[j%2]) frees V stage j%2, so the producers wait on those.
  static constexpr int bSFull = bVFull + VST;      // one per S buffer
  static constexpr int bPFull = bSFull + kNumS;     // one per S buffer (see below)
  static constexpr int bOReady = bPFull + kNumS;    // two, alternating by step parity
  static constexpr int bFin = bOReady + 2;
  static constexpr int kNumBars = bFin + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;   // tmem base, abort, n_entries
  static constexpr int kRed = kMisc + 64;             // [2 parities][2 halves][128] row maxima
  static constexpr int kLRed = kRed + 2 * 2 * BM * 4; // [2 halves][128] row sums
  static constexpr int kBits = kLRed + 2 * BM * 4;
  static constexpr int kInfo = kBits + 2 * (kMaxNbAttn / 32) * 4;
  static constexpr int kEnd = kInfo + kMaxNbAttn * 2;
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
  kSiteKEmpty = 0, kSiteVEmpty, kSiteQFull, kSiteKFull, kSitePFull, kSiteVFull,
  kSiteSFull, kSiteOReady, kSiteFin
};
__device__ __forceinline__ void note_timeout(int32_t* st, int site) {
  set_status(st, SA_DEV_TIMEOUT | (1 << (8 + site)));
}

// max over 64 fp32 values (bit patterns), eight independent chains.
__device__ __forceinline__ float max64(const uint32_t* v) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = __uint_as_float(v[i]);
#pragma unroll
  for (int i = 8; i < 64; ++i) m[i & 7] = fmaxf(m[i & 7], __uint_as_float(v[i]));
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}

// p = 2^(s * c - m) for 64 logits, packed as fp16 pairs into 32 words;
// returns the fp32 sum of the p (eight independent chains).
__device__ __forceinline__ float exp_pack64(const uint32_t* v, float c, float negm,
                                            uint32_t* pk) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
  for (int u = 0; u < 64; u += 2) {
    const float p0 = fast_exp2(fmaf(__uint_as_float(v[u]), c, negm));
    const float p1 = fast_exp2(fmaf(__uint_as_float(v[u + 1]), c, negm));
    acc[(u >> 1) & 7] += p0 + p1;
    pk[u >> 1] = pack_half2(p0, p1);
  }
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) acc[i] += acc[i + w];
  return acc[0];
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
  const int pair = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Nb = a.Nb, S = a.S;
  const int qb0 = 2 * pair;
  const bool has_qb1 = qb0 + 1 < Nb;

  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const AbortSignal abort_sig{abort_flag, a.dev_status};
  const volatile int never_flag = 0;
  const AbortSignal drain_sig{&never_flag, nullptr};  // drains wait out their own limit
  uint32_t* bmA = reinterpret_cast<uint32_t*>(smem + L::kBits);
  uint32_t* bmB = bmA + kMaxNbAttn / 32;
  uint16_t* info = reinterpret_cast<uint16_t*>(smem + L::kInfo);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    // p_full: every softmax thread arrives; the rest: one arrival (TMA
    // expect_tx or tcgen05.commit). There is one p_full per S buffer: the
    // softmax may finish several steps before the MMA thread looks, but the
    // next phase of p_full[j%3] needs QK(j+3), which the MMA thread issues
    // only after it has seen phase j, so a parity wait never falls a full
    // round behind. (The same holds for every other barrier here: none can
    // complete its next phase before its waiter has seen the current one.)
    for (int i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i >= L::bPFull && i < L::bPFull + kNumS) ? kSoftmaxThreads : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
    }
    // Union of the two query blocks' key lists, ascending, with a 2-bit
    // membership mask per key block: bit 0 = block 2p lists it, bit 1 = 2p+1.
    const int words = (Nb + 31) >> 5;
    int bad = 0;
    if (a.row_ptr == nullptr) {
      const uint16_t m = has_qb1 ? 3 : 1;
      for (int j = lane; j < Nb; j += 32) info[j] = static_cast<uint16_t>((j << 2) | m);
      if (lane == 0) misc[2] = static_cast<uint32_t>(Nb);
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
      int total = 0;
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
        int pos = total + incl - c;
        while (u) {
          const int bit = __ffs(u) - 1;
          const uint32_t m = ((ua >> bit) & 1u) | (((ub >> bit) & 1u) << 1);
          info[pos++] = static_cast<uint16_t>(((w * 32 + bit) << 2) | m);
          u &= u - 1;
        }
        total += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) misc[2] = static_cast<uint32_t>(total);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(a.dev_status, SA_DEV_BAD_ROUTE);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int n_entries = static_cast<int>(misc[2]);
  const int n_steps = (n_entries + 1) >> 1;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Lane 0 streams Q and then K, lane 1 streams V, each as far ahead as its
    // ring allows, so a K load never waits behind a V stage or vice versa.
    // Each lane waits for all of its own copies to land before it leaves, so
    // no copy can outlive the CTA's shared memory.
    if (lane == 0) {
      int issued[KST] = {0};
      bool ok = true;
      mbar_arrive_expect_tx(bar(L::bQFull), L::kQBytes);
      for (int qh = 0; qh < 2; ++qh)
        for (int dh = 0; dh < D / 64; ++dh)
          tma_load_4d(sbase + L::kQ + dh * L::kRegion + qh * 8192, &tm_q, bar(L::bQFull),
                      dh * 64, (qb0 + qh) * kBlock, h, b);
      for (int j = 0; j < n_steps; ++j) {
        const int nblk = (2 * j + 1 < n_entries) ? 2 : 1;
        const int ks = j % KST;
        if (j >= KST && !mbar_wait(bar(L::bSFull + ks), ((j / KST) - 1) & 1, abort_sig)) {
          note_timeout(a.dev_status, kSiteKEmpty);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::bKFull + ks), nblk * kBlock * D * 2);
        ++issued[ks];
        for (int kh = 0; kh < nblk; ++kh) {
          const int jk = info[2 * j + kh] >> 2;
          for (int dh = 0; dh < D / 64; ++dh)
            tma_load_4d(sbase + L::kK + ks * L::kKBytes + dh * L::kRegion + kh * 8192, &tm_k,
                        bar(L::bKFull + ks), dh * 64, jk * kBlock, h, b);
        }
      }
      if (!ok) *abort_flag = 1;
      mbar_wait(bar(L::bQFull), 0, drain_sig);
      for (int s2 = 0; s2 < KST; ++s2)
        if (issued[s2]) mbar_wait(bar(L::bKFull + s2), (issued[s2] - 1) & 1, drain_sig);
    } else if (lane == 1) {
      int issued[VST] = {0};
      bool ok = true;
      for (int j = 0; j < n_steps; ++j) {
        const int nblk = (2 * j + 1 < n_entries) ? 2 : 1;
        const int vs = j % VST;
        if (j >= VST && !mbar_wait(bar(L::bOReady + vs), ((j / VST) - 1) & 1, abort_sig)) {
          note_timeout(a.dev_status, kSiteVEmpty);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::bVFull + vs), nblk * kBlock * D * 2);
        ++issued[vs];
        for (int kh = 0; kh < nblk; ++kh) {
          const int jk = info[2 * j + kh] >> 2;
          tma_load_3d(sbase + L::kV + vs * L::kVBytes + kh * L::kVHalf, &tm_vt,
                      bar(L::bVFull + vs), jk * kBlock, 0, b * a.H + h);
        }
      }
      if (!ok) *abort_flag = 1;
      for (int s2 = 0; s2 < VST; ++s2)
        if (issued[s2]) mbar_wait(bar(L::bVFull + s2), (issued[s2] - 1) & 1, drain_sig);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t kIdQK128 = idesc_f16(BM, 128, 1);
      constexpr uint32_t kIdQK64 = idesc_f16(BM, 64, 1);
      constexpr uint32_t kIdPV = idesc_f16(BM, D, 0);
      // Q always lands before the CTA can exit, even with an empty route.
      bool ok = mbar_wait(bar(L::bQFull), 0, abort_sig);
      if (!ok) note_timeout(a.dev_status, kSiteQFull);
      // Descriptors: fixed high words, start addresses stepped in the low word.
      const uint64_t q_desc = sdesc_kmajor_sw128(sbase + L::kQ);
      const uint64_t k_desc = sdesc_kmajor_sw128(sbase + L::kK);
      const uint64_t v_desc = sdesc_kmajor_sw128(sbase + L::kV);
      const uint32_t desc_hi = static_cast<uint32_t>(q_desc >> 32);
      const uint32_t q_lo = static_cast<uint32_t>(q_desc);
      const uint32_t k_lo = static_cast<uint32_t>(k_desc);
      const uint32_t v_lo = static_cast<uint32_t>(v_desc);
      auto issue_qk = [&](int j) -> bool {
        const int ks = j % KST;
        if (!mbar_wait(bar(L::bKFull + ks), (j / KST) & 1, abort_sig)) {
          note_timeout(a.dev_status, kSiteKFull);
          return false;
        }
        tc_fence_after();
        const uint32_t idesc = (2 * j + 1 < n_entries) ? kIdQK128 : kIdQK64;
        const uint32_t d_tmem = tmem + (j % kNumS) * 128;
        const uint32_t kb = k_lo + ks * (L::kKBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kRegion + (kk & 3) * 32) >> 4;
          umma_ss_lohi(d_tmem, q_lo + off, desc_hi, kb + off, desc_hi, idesc, kk > 0);
        }
        umma_commit(bar(L::bSFull + (j % kNumS)));
        return true;
      };
      if (ok && n_steps > 0) tc_fence_after();
      for (int j = 0; j < kNumS && j < n_steps && ok; ++j) ok = issue_qk(j);
      for (int j = 0; j < n_steps && ok; ++j) {
        if (!mbar_wait(bar(L::bPFull + j % kNumS), (j / kNumS) & 1, abort_sig)) {
          note_timeout(a.dev_status, kSitePFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const int vs = j % VST;
        if (!mbar_wait(bar(L::bVFull + vs), (j / VST) & 1, abort_sig)) {
          note_timeout(a.dev_status, kSiteVFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = tmem + (j % kNumS) * 128;  // P(j) over S(j)
        const uint32_t vb = v_lo + vs * (L::kVBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts_lohi(tmem + kColO, pa + 8 * kk, vb + ((kk & 3) * 32 >> 4), desc_hi, kIdPV,
                       (j > 0 || kk > 0));
        if (2 * j + 1 < n_entries) {
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            umma_ts_lohi(tmem + kColO, pa + 8 * kk,
                         vb + ((L::kVHalf + (kk & 3) * 32) >> 4), desc_hi, kIdPV, 1u);
        }
        umma_commit(bar(L::bOReady + (j & 1)));
        // S[j%3] now belongs to QK(j+3): PV(j), the last reader of P(j), was
        // issued just before, and the tensor pipe runs this thread's MMAs in
        // order.
        if (j + kNumS < n_steps && !issue_qk(j + kNumS)) { ok = false; break; }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.dev_status, SA_DEV_TIMEOUT);
      }
      // Every MMA issued above completes before TMEM is released.
      umma_commit(bar(L::bFin));
      mbar_wait(bar(L::bFin), 0, drain_sig);
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Two threads per row: `half` 0 owns the step's first key block and O
    // columns [0, D/2); `half` 1 the second block and O columns [D/2, D).
    // The pair meets at named barrier 1 + quarter every step, so a thread
    // that gives up on a wait keeps looping (skipping all waits and TMEM
    // work) to keep the pair's barrier counts equal.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;         // tile row == TMEM lane
    const int qh = r >> 6;                     // query block of this row (warp-uniform)
    const int t = qb0 * kBlock + r;            // query token
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int last_valid = S - (Nb - 1) * kBlock;  // tokens in the last block
    const float cl2 = a.scale_log2;
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    float* lred = reinterpret_cast<float*>(smem + L::kLRed);
    const uint32_t pair_bar = 1 + quarter;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;

    for (int j = 0; j < n_steps; ++j) {
      if (ok && !mbar_wait_warp(bar(L::bSFull + j % kNumS), (j / kNumS) & 1, abort_sig)) {
        ok = false;
        if (lane == 0) note_timeout(a.dev_status, kSiteSFull);
      }
      if (ok) tc_fence_after();
      const int nblk = (2 * j + 1 < n_entries) ? 2 : 1;
      const bool present = half == 0 || nblk == 2;
      const uint32_t e = present ? info[2 * j + half] : 0u;
      const bool mem = ok && present && ((e >> qh) & 1u);
      const uint32_t s_col = (j % kNumS) * 128;

      uint32_t sr[64];
      float my_max = -INFINITY;
      if (mem) {
        tmem_ld32(lane_base + s_col + 64 * half, sr);
        tmem_ld32(lane_base + s_col + 64 * half + 32, sr + 32);
        tmem_wait_ld();
        if (static_cast<int>(e >> 2) == Nb - 1) {  // ragged last block: keys past S weigh 0
#pragma unroll
          for (int u = 0; u < 64; ++u)
            if (u >= last_valid) sr[u] = __float_as_uint(-INFINITY);
        }
        my_max = max64(sr);
      }
      float* slot = red + (j & 1) * 2 * BM;
      slot[half * BM + r] = my_max;
      // the partner's S loads are ordered before this thread's P stores,
      // which overwrite S columns 32-63 of the partner's half
      tc_fence_before();
      named_bar_sync(pair_bar, 64);
      tc_fence_after();
      const float mx = fmaxf(my_max, slot[(half ^ 1) * BM + r]);
      if (!ok) continue;
      const float bmax = mx * cl2;           // the scale is positive: max commutes
      float m_new = m_run;
      if (bmax > m_run + kRescaleLog2) m_new = bmax;  // also the first finite block
      const bool rescale = (m_new != m_run) && (m_run != -INFINITY);
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      // P(j) over the consumed S(j) columns: keys 0-63 -> columns 0-31,
      // keys 64-127 -> columns 32-63 (two fp16 per column).
      float rs = 0.f;
      if (present) {
        uint32_t pk[32];
        if (mem) rs = exp_pack64(sr, cl2, -m_new, pk);
        else {
#pragma unroll
          for (int u = 0; u < 32; ++u) pk[u] = 0u;
        }
        tmem_st32(lane_base + s_col + 32 * half, pk);
      }
      l_run = l_run * alpha + rs;
      m_run = m_new;
      if (__any_sync(0xffffffffu, rescale)) {
        // PV(j-1) must be done before O is scaled (j > 0 here: m_run was
        // finite). S(j) ready implies PV(j-3) done (QK(j) was issued after
        // it) and PV(j+1) is not yet issued, so on the barrier of PV(j-1)'s
        // parity the phase of PV(j-1) is either the last completed or the
        // pending one: no ambiguity.
        if (!mbar_wait_warp(bar(L::bOReady + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_sig)) {
          ok = false;
          if (lane == 0) note_timeout(a.dev_status, kSiteOReady);
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          const uint32_t col = kColO + half * (D / 2) + 32 * c;
          tmem_ld32(lane_base + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          tmem_st32(lane_base + col, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::bPFull + j % kNumS));
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(a.dev_status, SA_DEV_TIMEOUT);
    }

    // ------------------------------------------------------------ epilogue
    lred[half * BM + r] = l_run;
    named_bar_sync(pair_bar, 64);
    const float l_tot = l_run + lred[(half ^ 1) * BM + r];
    bool have_o = ok && n_steps > 0;
    if (have_o) {
      // The MMA thread commits bFin after its last PV; softmax need not have
      // seen every o_ready phase, so that barrier's parity is no guide here.
      have_o = mbar_wait_warp(bar(L::bFin), 0, abort_sig);
      if (!have_o) {
        *abort_flag = 1;
        if (lane == 0) note_timeout(a.dev_status, kSiteFin);
      }
      tc_fence_after();
    }
    const bool row_ok = t < S;
    const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
    uint16_t* orow = a.o + b * a.os[0] + static_cast<int64_t>(t) * a.os[1] + h * a.os[2] +
                     half * (D / 2);
    uint32_t o[D / 2];
    if (have_o) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(lane_base + kColO + half * (D / 2) + 32 * c, o + 32 * c);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int u = 0; u < D / 2; ++u) o[u] = 0u;
    }
    if (row_ok) {
#pragma unroll
      for (int v = 0; v < D / 16; ++v) {
        uint4 w;
        w.x = pack_bf162(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
        w.y = pack_bf162(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
        w.z = pack_bf162(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
        w.w = pack_bf162(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
        *reinterpret_cast<uint4*>(orow + 8 * v) = w;
      }
    }
    if (row_ok && half == 0 && a.lse) {
      const float lse = l_tot > 0.f ? m_run * 0.69314718055994531f + logf(l_tot) : -INFINITY;
      a.lse[(static_cast<int64_t>(b) * a.H + h) * S + t] = lse;
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
  dim3 grid(a.n_pairs, a.H, a.B);
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
