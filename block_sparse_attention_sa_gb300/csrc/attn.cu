// attn.cu -- block-sparse flash-attention forward on sm_103a (tcgen05/TMEM/TMA).
//
// What is computed: for every query token of 64-token block i, exact softmax
// attention over the valid tokens of the key blocks routed to (b, h, i)
// (MiniAcc blog, "What is Sol attention?": only the selected pairs are
// computed; "MiniMax H3 runs on single 4090 with 4.44x speedup over dense
// execution", third paragraph: the exact prefix sink and the diagonal are
// part of every route). Dense mode lists every key block.
//
// Tiles. A tile is a 128-row query tile = two 64-token query blocks of one
// head (tcgen05 M = 128; the route is per 64-row block). Its key walk is the
// union of the two blocks' key lists, two 64-key blocks per step (N = 128);
// a key block listed for only one of the two query blocks is masked to -inf
// for the other half's rows, so each row still sees exactly its own key set.
// The walk starts at the tile's diagonal block, where row maxima usually are.
//
// Persistent CTAs. One CTA per SM takes tiles from a global counter in
// (batch, head, pair) order, so concurrently running tiles share a head's
// K/V in L2. While one tile runs, a planner warp builds the next tile's key
// walk into the other half of a double buffer, and the next tile's first
// QK^T products are computed during the current tile's epilogue.
//
// Pipeline. TMEM holds three S buffers and one O accumulator (3 x 128 + D
// columns). Step j's S = Q K(j)^T (bf16 x bf16 -> fp32) goes to buffer j % 3;
// the softmax turns it into P (fp16) over the same columns; O += P V(j)
// (fp16, A from TMEM). The MMA warp issues QK^T(j+2) before it waits for
// P(j) -- its buffer last held step j-1, whose PV was issued already -- so
// the tensor pipe has the next products queued while the softmax works.
//
// Softmax. Two warpgroups take the steps in turn (warpgroup 0 the even
// steps of this CTA's sequence, warpgroup 1 the odd ones), one thread per
// row with all 128 keys of its step, so each warpgroup has two steps' time
// for one step's chain. The rows' running max passes from step to step
// through shared memory: a thread publishes the max after its step as soon
// as it knows it, and the thread of the next step reads it before its
// exponentials (it seldom waits: the previous step started a whole step
// earlier). Each warpgroup keeps its own partial row sum; the two threads of
// a row add them in the epilogue. The running max moves only when a block
// max exceeds it by more than 2^14 (then O is rescaled, after the last PV
// into it has completed). The block maxima come with the S loads themselves
// (the reduction form of tcgen05.ld returns each 32-column maximum), so the
// chain from S to the exponentials holds no maximum instructions of its own
// except in the ragged last key block, which is masked first.
//
// Warps: 0-3 softmax of even steps, 4-7 of odd steps, 8 producer (Q, and K and
// V through one ring of stages in the order the MMA warp consumes them),
// 9 MMA (converged; elect.sync issues), 10 planner, 11 idle. No
// data-dependent load sits inside a pipelined loop: the walk is built ahead
// by the planner. Every wait is bounded (SA_DEV_TIMEOUT); the two threads of
// a row carry a stop bit through both of their exchanges so they always
// leave together, and an aborted CTA drains its own copies and MMAs and
// frees TMEM before it exits.
#include <climits>
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sa_internal.cuh"

namespace sa {

namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // key rows per step (two key blocks)
constexpr int KVST = 5;   // stages of the K/V ring (each holds one K or one V^T tile of a step)
constexpr int kSBuf = 3;  // S buffers in TMEM
constexpr int kSets = 2;  // softmax warpgroups, taking the steps in turn
constexpr int kThreads = 384;        // three warpgroups: softmax (two), control
constexpr int kSetThreads = 128;     // one softmax thread per row and warpgroup
constexpr int kSoftmaxThreads = kSets * kSetThreads;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kPlannerWarp = 10;  // warp 11: barriers only
// Register split (setmaxnreg). At launch ptxas gives every thread
// kLaunchRegs (65536 / 384 rounded down to a multiple of 8); the two softmax
// warpgroups then grow to kSoftmaxRegs and the control warpgroup shrinks
// to kControlRegs: 2*128*216 + 128*64 = 63,488 <= 384*168 = 64,512, and per
// SM sub-partition (one warp of each warpgroup) 216 + 216 + 64 <= 512. A
// softmax thread holds a whole 128-key row of S (128 registers) at once.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 216;
constexpr int kControlRegs = 64;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;
constexpr int kColS = 0;      // S[b] at columns [128 b, 128 b + 128), b < kSBuf
constexpr int kColO = 384;    // O at columns [384, 384 + D)
// Lazy rescale: the running max moves only when a block max exceeds it by
// more than 2^14, so P <= 16384 stays well inside fp16; values that fall
// below fp16's normal range weigh under 2^-28 of the row max.
constexpr float kRescaleLog2 = 14.0f;

template <int D, bool kF8>
struct Smem {
  static constexpr int kRegion = BM * 128;            // one 128-byte-wide K slice of 128 rows
  static constexpr int kQ = 0;
  static constexpr int kQBytes = BM * D * (kF8 ? 1 : 2);  // bf16, or e4m3 codes
  static constexpr int kQKSlices = kF8 ? D / 128 : D / 64;  // 128-byte slices of a Q/K row
  static constexpr int kStageBytes = BN * D * 2;      // one K tile or one V^T tile of a step
  static constexpr int kKV = kQ + kQBytes;
  static constexpr int kVHalf = D * 128;              // one 64-key half of a V^T tile
  static constexpr int kBar = kKV + KVST * kStageBytes;
  // barriers (counts in the init loop below)
  static constexpr int bInfoFull = 0;                 // [2] planner wrote walk x
  static constexpr int bInfoEmpty = bInfoFull + 2;    // [2] every consumer is done with walk x
  static constexpr int bQFull = bInfoEmpty + 2;       // Q of the current tile landed
  static constexpr int bQEmpty = bQFull + 1;          // the tile's last QK is done with Q
  static constexpr int bKVFull = bQEmpty + 1;         // [KVST] a stage landed
  static constexpr int bKVEmpty = bKVFull + KVST;     // [KVST] its MMAs are done with a stage
  static constexpr int bSFull = bKVEmpty + KVST;      // [kSBuf] QK into S[b] done
  static constexpr int bPFull = bSFull + kSBuf;       // [kSBuf] softmax wrote P over S[b]
  static constexpr int bPVDone = bPFull + kSBuf;      // [2] PV number g (this CTA's count)
                                                      // completes a phase of bPVDone + g % 2
  static constexpr int bTileDone = bPVDone + 2;       // every PV of the tile done
  static constexpr int bOFree = bTileDone + 1;        // the epilogue has read O
  static constexpr int bFin = bOFree + 1;             // every MMA done (exit)
  static constexpr int kNumBars = bFin + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;   // tmem base, abort flag
  // [2][8] walk headers: b, h, pair, n, and (8-bit scores) the scale
  // exponents of the tile's two query blocks
  static constexpr int kHdr = kMisc + 16;
  // row exchange: [2 slots][2 warpgroups][BM] of (m, l, stop)
  static constexpr int kXch = kHdr + 64;
  static constexpr int kXchBytes = 2 * kSets * BM * 12;
  // running-max handoff: [2 warpgroups][BM] max after the warpgroup's latest
  // step, and that step's index in the CTA's sequence
  static constexpr int kHand = kXch + kXchBytes;
  static constexpr int kHandBytes = kSets * BM * 8;
  static constexpr int kBits = kHand + kHandBytes;
  static constexpr int kInfo = kBits + 2 * (kMaxNbAttn / 32) * 4;  // [2][kMaxNbAttn] walks
  static constexpr int kKexp = kInfo + 2 * kMaxNbAttn * 2;  // [2][kMaxNbAttn] key-block
                                                            // scale exponents of the walks
  static constexpr int kEnd = kKexp + (kF8 ? 2 * kMaxNbAttn : 0);
  static constexpr int kBytes = kEnd + 1024;          // slack to align the base to 1 KB
  static_assert(kBar % 8 == 0 && kMisc % 8 == 0 && kHdr % 4 == 0 && kXch % 4 == 0,
                "barrier, header and exchange alignment");
  static_assert(kHand % 8 == 0 && kBits % 4 == 0 && kInfo % 2 == 0,
                "shared-memory region alignment");
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
  kSiteKVStage = 0, kSiteQFull, kSiteKVFull, kSitePFull, kSiteSFull, kSiteFin, kSiteInfo,
  kSiteOFree, kSitePVDone, kSiteHandoff
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

// max over 32 fp32 values (bit patterns): four chains of three-input max.
__device__ __forceinline__ float max32(const uint32_t* v) {
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmaxf(__uint_as_float(v[i]), __uint_as_float(v[4 + i]));
#pragma unroll
  for (int i = 8; i < 32; i += 8)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      m[c] = fmax3(m[c], __uint_as_float(v[i + c]), __uint_as_float(v[i + 4 + c]));
  return fmax3(fmaxf(m[0], m[1]), m[2], m[3]);
}

// p = 2^(s * c - m) for 32 logits, packed as fp16 pairs into 16 words;
// returns the fp32 sum of the p (paired fp32 arithmetic, four sum chains).
__device__ __forceinline__ float exp_pack32(const uint32_t* v, float c, float negm,
                                            uint32_t* pk) {
  const uint64_t c2 = f2_pack(c, c), m2 = f2_pack(negm, negm);
  uint64_t acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0ull;
#pragma unroll
  for (int u = 0; u < 32; u += 2) {
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

// Keys [32 half, 32 half + 32) of a key block: in the ragged last block the
// logits of keys past S become -inf (weight 0).
__device__ __forceinline__ void mask_tail32(uint32_t* v, uint32_t entry, int half, int Nb,
                                            int last_valid) {
  if (static_cast<int>(entry >> 2) == Nb - 1) {
#pragma unroll
    for (int u = 0; u < 32; ++u)
      if (u + 32 * half >= last_valid) v[u] = __float_as_uint(-INFINITY);
  }
}

template <int D, bool kF8>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_vt, const AttnArgs a) {
  using L = Smem<D, kF8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nb = a.Nb, S = a.S;
  const unsigned full = 0xffffffffu;

  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const AbortSignal abort_sig{abort_flag, a.grid_abort};
  const volatile int never_flag = 0;
  const AbortSignal drain_sig{&never_flag, nullptr};  // drains wait out their own limit
  volatile int* hdr = reinterpret_cast<volatile int*>(smem + L::kHdr);
  uint16_t* info = reinterpret_cast<uint16_t*>(smem + L::kInfo);
  int8_t* kexp = reinterpret_cast<int8_t*>(smem + L::kKexp);   // used with kF8 only
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  auto fail = [&](int site) {
    *abort_flag = 1;
    if (a.grid_abort) *reinterpret_cast<volatile int*>(a.grid_abort) = 1;
    note_timeout(a.dev_status, site);
  };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    // Arrival counts. No barrier can complete its next phase before each of
    // its waiters has seen the current one, so parity waits never fall a
    // full round behind: every next phase needs work the waiter releases
    // after its wait (the walk buffers need all their consumers; a ring
    // stage is refilled only after its MMAs freed it, and they wait for it
    // to fill; QK into S[b] again needs the PV that read P(b), which waits
    // for p_full; a PV-done phase needs a PV, which needs the softmax's
    // p_full; the next tile's first PV waits for o_free, which needs every
    // softmax thread past its tile_done wait; and so on).
    for (int i = 0; i < L::kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == L::bInfoEmpty || i == L::bInfoEmpty + 1) cnt = 2 + kSoftmaxThreads;
      if (i >= L::bPFull && i < L::bPFull + kSBuf) cnt = kSetThreads;
      if (i == L::bOFree) cnt = kSoftmaxThreads;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < kSoftmaxThreads)   // no step published yet (index -1)
    reinterpret_cast<uint64_t*>(smem + L::kHand)[threadIdx.x] = 0xffffffff00000000ull;
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
    // A route that breaks the CSR contract raises SA_DEV_BAD_ROUTE: a row
    // whose span is not inside [0, nnz] or longer than Nb is skipped whole,
    // an entry outside [0, Nb) is skipped, and a row that is not strictly
    // ascending (a duplicate included) is attended as the set of its entries.
    uint32_t* bmA = reinterpret_cast<uint32_t*>(smem + L::kBits);
    uint32_t* bmB = bmA + kMaxNbAttn / 32;
    const int nnz = a.row_ptr != nullptr ? a.row_ptr[a.nnz_row] : 0;
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
      volatile int* hd = hdr + 8 * x;
      uint16_t* inf = info + x * kMaxNbAttn;
      int8_t* kx = kexp + x * kMaxNbAttn;
      if (tile >= a.n_tiles) {
        if (lane == 0) hd[3] = -1;   // no more tiles: every role leaves its loop
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bInfoFull + x));
        break;
      }
      const int slot = tile % a.n_pairs;
      const int bh = tile / a.n_pairs;
      const int h = bh % a.H, b = bh / a.H;
      // the tile's two query blocks qb0 < qb1 (qb1 = -1: qb0 alone)
      int qb0 = 2 * slot, qb1 = qb0 + 1 < Nb ? qb0 + 1 : -1;
      int bad = 0;
      if (a.pairs) {
        const uint32_t pe = a.pairs[static_cast<int64_t>(bh) * a.n_pairs + slot];
        qb0 = static_cast<int>(pe & 0xffffu);
        qb1 = (pe >> 16) == 0xffffu ? -1 : static_cast<int>(pe >> 16);
        if (qb0 >= Nb || qb1 >= Nb || qb1 == qb0) {   // never written by the pairing kernels
          bad = 1;
          qb0 = 0;
          qb1 = -1;
        }
      }
      const bool has_qb1 = qb1 >= 0;
      // Union of the two query blocks' key lists with a 2-bit membership mask
      // per key block (bit 0: block qb0 lists it, bit 1: block qb1 does),
      // ascending but rotated to start at the tile's own diagonal block: the
      // row maxima usually sit near the diagonal, so taking it first keeps
      // later steps from raising the running max (each raise rescales O).
      const int words = (Nb + 31) >> 5;
      if (a.row_ptr == nullptr) {
        const uint16_t m = has_qb1 ? 3 : 1;
        for (int j = lane; j < Nb; j += 32) {
          inf[(j - qb0 + Nb) % Nb] = static_cast<uint16_t>((j << 2) | m);
          if (kF8) kx[(j - qb0 + Nb) % Nb] = a.k_exp[static_cast<int64_t>(bh) * Nb + j];
        }
        if (lane == 0) hd[3] = Nb;
      } else {
        for (int w = lane; w < words; w += 32) { bmA[w] = 0u; bmB[w] = 0u; }
        __syncwarp();
        for (int half = 0; half < 2; ++half) {
          if (half == 1 && !has_qb1) break;
          const int64_t r = (static_cast<int64_t>(b) * a.H + h) * Nb + (half ? qb1 : qb0);
          const int beg = a.row_ptr[r], end = a.row_ptr[r + 1];
          if (beg < 0 || end < beg || end - beg > Nb || end > nnz) { bad = 1; continue; }
          uint32_t* bm = half ? bmB : bmA;
          int carry = INT_MIN;                 // the entry before this chunk
          for (int e0 = beg; e0 < end; e0 += 32) {
            const int e = e0 + lane;
            const bool in = e < end;
            const int j = in ? a.col_idx[e] : INT_MAX;
            int prev = __shfl_up_sync(full, j, 1);
            if (lane == 0) prev = carry;
            if (in && prev >= j) bad = 1;      // not strictly ascending
            if (in) {
              if (j < 0 || j >= Nb) bad = 1;
              else atomicOr(&bm[j >> 5], 1u << (j & 31));
            }
            carry = __shfl_sync(full, j, 31);
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
            if (kF8) kx[rp] = a.k_exp[static_cast<int64_t>(bh) * Nb + w * 32 + bit];
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
        hd[2] = static_cast<int>(static_cast<uint32_t>(qb0) | (static_cast<uint32_t>(qb1 & 0xffff) << 16));
        if (kF8) {
          hd[4] = a.q_exp[static_cast<int64_t>(bh) * Nb + qb0];
          hd[5] = has_qb1 ? a.q_exp[static_cast<int64_t>(bh) * Nb + qb1] : 0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bInfoFull + x));
    }
  } else if (warp == kProducerWarp) {
    regs_dec<kControlRegs>();
    // ------------------------------------------------------------- producer
    // Lane 0 loads each tile's Q, and K and V^T tiles through the ring in the
    // order the MMA warp consumes them: K(0), K(1), then K(j+2) and V(j) for
    // each step j (2 * n_steps items per tile). A stage is refilled once the
    // MMAs that read it are done. The lane waits for all of its own copies to
    // land before it leaves, so no copy can outlive the CTA's shared memory.
    if (lane == 0) {
      int issued[KVST] = {0};
      int q_loads = 0, c = 0;
      for (int it = 0;; ++it) {
        const int x = it & 1;
        if (!mbar_wait(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) { fail(kSiteInfo); break; }
        const volatile int* hd = hdr + 8 * x;
        const int n = hd[3];
        if (n < 0) break;
        const int b = hd[0], h = hd[1];
        // query rows of the two blocks; a missing second block reads zeros
        const uint32_t pr = static_cast<uint32_t>(hd[2]);
        const int qrow0 = static_cast<int>(pr & 0xffffu) * kBlock;
        const int qrow1 = (pr >> 16) == 0xffffu ? Nb * kBlock : static_cast<int>(pr >> 16) * kBlock;
        const int bh = b * a.H + h;
        const uint16_t* inf = info + x * kMaxNbAttn;
        // the previous tile's QKs are done with the Q buffer
        if (it >= 1 && !mbar_wait(bar(L::bQEmpty), (it - 1) & 1, abort_sig)) { fail(kSiteQFull); break; }
        mbar_arrive_expect_tx(bar(L::bQFull), L::kQBytes);
        ++q_loads;
        for (int qh = 0; qh < 2; ++qh)
          for (int dh = 0; dh < L::kQKSlices; ++dh)
            tma_load_4d(sbase + L::kQ + dh * L::kRegion + qh * 8192, &tm_q, bar(L::bQFull),
                        dh * 64, qh ? qrow1 : qrow0, h, b);
        const int n_steps = (n + 1) >> 1;
        // one ring item: K (kind 0) or V^T (kind 1) of step js
        auto load_item = [&](int kind, int js) -> bool {
          const int st = c % KVST;
          if (c >= KVST && !mbar_wait(bar(L::bKVEmpty + st), ((c / KVST) - 1) & 1, abort_sig)) {
            fail(kSiteKVStage);
            return false;
          }
          const int nblk = (2 * js + 1 < n) ? 2 : 1;
          mbar_arrive_expect_tx(bar(L::bKVFull + st),
                                nblk * kBlock * D * ((kF8 && kind == 0) ? 1 : 2));
          ++issued[st];
          const uint32_t dst = sbase + L::kKV + st * L::kStageBytes;
          for (int kh = 0; kh < nblk; ++kh) {
            const int jk = inf[2 * js + kh] >> 2;
            if (kind == 0) {
              for (int dh = 0; dh < L::kQKSlices; ++dh)
                tma_load_4d(dst + dh * L::kRegion + kh * 8192, &tm_k, bar(L::bKVFull + st),
                            dh * 64, jk * kBlock, h, b);
            } else {
              tma_load_3d(dst + kh * L::kVHalf, &tm_vt, bar(L::bKVFull + st), jk * kBlock, 0, bh);
            }
          }
          ++c;
          return true;
        };
        bool ok = true;
        if (n_steps > 0) ok = load_item(0, 0);
        if (ok && n_steps > 1) ok = load_item(0, 1);
        for (int j = 0; j < n_steps && ok; ++j) {
          if (j + 2 < n_steps) ok = load_item(0, j + 2);
          if (ok) ok = load_item(1, j);
        }
        if (!ok) break;
        mbar_arrive(bar(L::bInfoEmpty + x));
      }
      if (q_loads) mbar_wait(bar(L::bQFull), (q_loads - 1) & 1, drain_sig);
      for (int s2 = 0; s2 < KVST; ++s2)
        if (issued[s2]) mbar_wait(bar(L::bKVFull + s2), (issued[s2] - 1) & 1, drain_sig);
    }
  } else if (warp == kMmaWarp) {
    regs_dec<kControlRegs>();
    // ------------------------------------------------------------------ MMA
    // The whole warp runs this loop in step (warp-uniform waits); elect.sync
    // picks the lane that issues each batch of MMAs and each commit (lane 0
    // of the converged warp, so every commit tracks every earlier MMA). Order
    // per tile: QK(0), QK(1), then for each step j: QK(j+2) (if any), PV(j)
    // -- the same order in which the producer fills the ring.
    constexpr uint32_t kIdQK128 = kF8 ? idesc_e4m3(BM, 128) : idesc_f16(BM, 128, 1);
    constexpr uint32_t kIdQK64 = kF8 ? idesc_e4m3(BM, 64) : idesc_f16(BM, 64, 1);
    // K slices of one MMA: 16 bf16 or 32 e4m3 values, 32 bytes either way
    constexpr int kKS = kF8 ? D / 32 : D / 16;
    constexpr uint32_t kIdPV = idesc_f16(BM, D, 0);
    // Descriptors: Q's K slices (start address stepped by 32 bytes inside a
    // 128-byte swizzle row, then by one 16 KB region per 64 elements), and
    // the ring's base.
    uint64_t qd[kKS];
#pragma unroll
    for (int kk = 0; kk < kKS; ++kk)
      qd[kk] = sdesc_kmajor_sw128(sbase + L::kQ + (kk >> 2) * L::kRegion + (kk & 3) * 32);
    const uint64_t kv0 = sdesc_kmajor_sw128(sbase + L::kKV);
    const uint32_t o_tmem = tmem + kColO;
    int c = 0;        // ring items consumed so far
    int gs0 = 0;      // global index (over this CTA's tiles) of the tile's first step
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int x = it & 1;
      if (!mbar_wait_warp(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig)) {
        if (lane == 0) fail(kSiteInfo);
        break;
      }
      const int n = hdr[8 * x + 3];
      if (n < 0) break;
      const int n_steps = (n + 1) >> 1;
      if (!mbar_wait_warp(bar(L::bQFull), it & 1, abort_sig)) {
        if (lane == 0) fail(kSiteQFull);
        break;
      }
      tc_fence_after();
      // QK(j) into S[(gs0 + j) % 3]. That buffer last held step gs0 + j - 3,
      // whose PV -- the last reader of its P -- this warp issued earlier; the
      // tensor pipe runs the MMAs in order.
      auto issue_qk = [&](int j) -> bool {
        const int st = c % KVST;
        if (!mbar_wait_warp(bar(L::bKVFull + st), (c / KVST) & 1, abort_sig)) {
          if (lane == 0) fail(kSiteKVFull);
          return false;
        }
        tc_fence_after();
        const int b = (gs0 + j) % kSBuf;
        const uint32_t idesc = (2 * j + 1 < n) ? kIdQK128 : kIdQK64;
        const uint32_t d_tmem = tmem + kColS + b * 128;
        const uint64_t kb = kv0 + static_cast<uint64_t>(st * (L::kStageBytes >> 4));
        uint64_t kd[kKS];
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk)
          kd[kk] = kb + static_cast<uint64_t>(((kk >> 2) * L::kRegion + (kk & 3) * 32) >> 4);
#pragma unroll
        for (int h4 = 0; h4 < kKS / 4; ++h4) {
          if (kF8)
            umma_ss_x4_f8_elect(d_tmem, qd[4 * h4], qd[4 * h4 + 1], qd[4 * h4 + 2],
                                qd[4 * h4 + 3], kd[4 * h4], kd[4 * h4 + 1], kd[4 * h4 + 2],
                                kd[4 * h4 + 3], idesc, h4 > 0);
          else
            umma_ss_x4_elect(d_tmem, qd[4 * h4], qd[4 * h4 + 1], qd[4 * h4 + 2], qd[4 * h4 + 3],
                             kd[4 * h4], kd[4 * h4 + 1], kd[4 * h4 + 2], kd[4 * h4 + 3], idesc,
                             h4 > 0);
        }
        umma_commit_elect(bar(L::bSFull + b));
        umma_commit_elect(bar(L::bKVEmpty + st));
        if (j == n_steps - 1) umma_commit_elect(bar(L::bQEmpty));  // Q no longer read
        ++c;
        return true;
      };
      // The previous tile's epilogue must have read O before this tile's
      // first PV overwrites it. The wait sits right before that PV, so the
      // epilogue overlaps this tile's first three Q.K^T products (an empty
      // tile waits before its tile_done, so that barrier never runs a phase
      // ahead of the epilogue that waits on it).
      auto wait_o_free = [&]() -> bool {
        if (it >= 1 && !mbar_wait_warp(bar(L::bOFree), (it - 1) & 1, abort_sig)) {
          if (lane == 0) fail(kSiteOFree);
          return false;
        }
        tc_fence_after();
        return true;
      };
      if (n_steps == 0) {
        umma_commit_elect(bar(L::bQEmpty));
        ok = wait_o_free();
      }
      for (int j = 0; j < 2 && j < n_steps && ok; ++j) ok = issue_qk(j);
      if (!ok) break;
      for (int j = 0; j < n_steps && ok; ++j) {
        // QK(j+2) needs no softmax result, so it goes first: the tensor pipe
        // works on it while this warp waits for P(j).
        if (j + 2 < n_steps && !issue_qk(j + 2)) {
          ok = false;
          break;
        }
        if (j == 0 && !wait_o_free()) {
          ok = false;
          break;
        }
        const int gsj = gs0 + j, b = gsj % kSBuf, st = c % KVST;
        bool unused = false;
        if (!mbar_wait2_warp(bar(L::bPFull + b), (gsj / kSBuf) & 1, bar(L::bKVFull + st),
                             (c / KVST) & 1, false, 0u, 0u, &unused, abort_sig)) {
          if (lane == 0) fail(kSitePFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = tmem + kColS + b * 128;    // P(j) over S(j)
        const uint64_t vb = kv0 + static_cast<uint64_t>(st * (L::kStageBytes >> 4));
        umma_ts_x4_elect(o_tmem, pa, vb, vb + 2, vb + 4, vb + 6, kIdPV, j > 0);
        if (2 * j + 1 < n) {
          const uint64_t vh = vb + (L::kVHalf >> 4);
          umma_ts_x4_elect(o_tmem, pa + 32, vh, vh + 2, vh + 4, vh + 6, kIdPV, 1u);
        }
        umma_commit_elect(bar(L::bKVEmpty + st));
        umma_commit_elect(bar(L::bPVDone + (gsj & 1)));
        ++c;
      }
      gs0 += n_steps;
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
    const int sm = warp >> 2;                  // warpgroup: steps g with g % 2 == sm
    const int quarter = warp & 3;              // TMEM lane quarter
    const int r = quarter * 32 + lane;         // tile row == TMEM lane
    const int qh = r >> 6;                     // query block of this row (warp-uniform)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t pair_bar = 1 + quarter;     // named barrier of warps quarter, quarter + 4
    const int last_valid = S - (Nb - 1) * kBlock;  // tokens in the last block
    const float cl2 = a.scale_log2;
    float* xm = reinterpret_cast<float*>(smem + L::kXch);      // [2 slots][2 warpgroups][BM]
    float* xl = xm + 2 * kSets * BM;
    int* xs = reinterpret_cast<int*>(xl + 2 * kSets * BM);
    // running-max handoff: (step index << 32) | max bits, one 64-bit word
    // per row and warpgroup, written and read whole
    volatile uint64_t* hand = reinterpret_cast<volatile uint64_t*>(smem + L::kHand);
    volatile uint64_t* hand_mine = hand + sm * BM + r;
    const volatile uint64_t* hand_theirs = hand + (sm ^ 1) * BM + r;
    int xc = 0;                                // exchanges so far (slot xc & 1)
    // Swap (m, l) and a stop bit with the other warpgroup's thread of this
    // row. Both threads pass the same sequence of exchanges (two per tile),
    // and a stop from either ends both, so neither is ever left waiting at
    // the pair barrier. Slots alternate: a slot is rewritten only after the
    // next exchange, which the partner reaches after reading it.
    auto pair_xchg = [&](float m, float l, bool stop, float& m_o, float& l_o) -> bool {
      const int sl = xc & 1;
      ++xc;
      const int mine = (sl * kSets + sm) * BM + r, theirs = (sl * kSets + (sm ^ 1)) * BM + r;
      xm[mine] = m;
      xl[mine] = l;
      xs[mine] = stop ? 1 : 0;
      named_bar_sync(pair_bar, 64);
      m_o = xm[theirs];
      l_o = xl[theirs];
      return stop || xs[theirs] != 0;
    };
    // Waits (bounded, like every wait here) until the other warpgroup has
    // published the running max after step g_prev for this warp's rows.
    auto wait_handoff = [&](int g_prev, uint64_t& hv) -> bool {
      hv = *hand_theirs;
      if (__all_sync(full, static_cast<int>(hv >> 32) >= g_prev)) return true;
      unsigned long long t0 = 0;
      if (lane == 0) t0 = globaltimer();
      for (uint32_t i = 1;; ++i) {
        hv = *hand_theirs;
        if (__all_sync(full, static_cast<int>(hv >> 32) >= g_prev)) return true;
        if ((i & 63u) == 0u) {
          int give_up = 0;
          if (lane == 0) give_up = abort_sig.raised() || (globaltimer() - t0 > kWaitTimeoutNs);
          if (__shfl_sync(full, give_up, 0)) return false;
        }
      }
    };
    int gs = 0;                                // steps of this CTA's earlier tiles

    for (int it = 0;; ++it) {
      const int x = it & 1;
      bool stop = !mbar_wait_warp(bar(L::bInfoFull + x), (it >> 1) & 1, abort_sig);
      if (stop && lane == 0) fail(kSiteInfo);
      float u0, u1;
      if (pair_xchg(0.f, 0.f, stop, u0, u1)) break;
      const volatile int* hd = hdr + 8 * x;
      const int n = hd[3];
      if (n < 0) break;
      const int b = hd[0], h = hd[1];
      const uint32_t pr = static_cast<uint32_t>(hd[2]);
      const int8_t* kx = kexp + x * kMaxNbAttn;
      const int eq = kF8 ? hd[4 + qh] : 0;     // the row's query-block scale exponent
      const int qb = qh ? ((pr >> 16) == 0xffffu ? -1 : static_cast<int>(pr >> 16))
                        : static_cast<int>(pr & 0xffffu);
      const uint16_t* inf = info + x * kMaxNbAttn;
      const int n_steps = (n + 1) >> 1;
      const int t = qb * kBlock + (r & (kBlock - 1));   // query token (< 0: no block)
      // m_run: the max this warpgroup's latest step of the tile used (the
      // scale of l_run, its partial row sum)
      float m_run = -INFINITY, l_run = 0.f;

      for (int j = (gs ^ sm) & 1; j < n_steps; j += kSets) {
        const int g = gs + j, sb = g % kSBuf;
        const uint32_t s_col = kColS + sb * 128;
        // the step's walk entries (and with 8-bit scores its scale factors)
        // do not depend on S: read them before waiting for it
        const bool two = 2 * j + 1 < n;             // an odd walk's last step has one block
        const uint32_t e0 = inf[2 * j], e1 = two ? inf[2 * j + 1] : 0u;
        const bool mem0 = (e0 >> qh) & 1u, mem1 = two && ((e1 >> qh) & 1u);
        // the loads also return each 32-column maximum; the ragged last key
        // block is masked first and takes its maximum in software
        const bool tail0 = static_cast<int>(e0 >> 2) == Nb - 1;
        const bool tail1 = two && static_cast<int>(e1 >> 2) == Nb - 1;
        // exp2-domain factor of each key block's logits: the softmax scale,
        // times 2^(e_q + e_k) with 8-bit scores (exact: powers of two)
        const float c0 = kF8 ? ldexpf(cl2, eq + kx[2 * j]) : cl2;
        const float c1 = kF8 ? (two ? ldexpf(cl2, eq + kx[2 * j + 1]) : cl2) : cl2;
        if (!mbar_wait_warp(bar(L::bSFull + sb), (g / kSBuf) & 1, abort_sig)) {
          if (lane == 0) fail(kSiteSFull);
          stop = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
        float hm0 = -INFINITY, hm1 = -INFINITY, hm2 = -INFINITY, hm3 = -INFINITY;
        if (mem0) {
          tmem_ld32_max(lane_base + s_col, sr, hm0);
          tmem_ld32_max(lane_base + s_col + 32, sr + 32, hm1);
        }
        if (mem1) {
          tmem_ld32_max(lane_base + s_col + 64, sr + 64, hm2);
          tmem_ld32_max(lane_base + s_col + 96, sr + 96, hm3);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
        if (mem0 || mem1) {
          tmem_wait_ld();
          if (mem0) {
            reg_fence32(sr);
            reg_fence32(sr + 32);
            reg_fence_f(hm0);
            reg_fence_f(hm1);
            if (tail0) {
              mask_tail32(sr, e0, 0, Nb, last_valid);
              mask_tail32(sr + 32, e0, 1, Nb, last_valid);
              mx0 = fmaxf(max32(sr), max32(sr + 32));
            } else {
              mx0 = fmaxf(hm0, hm1);
            }
          }
          if (mem1) {
            reg_fence32(sr + 64);
            reg_fence32(sr + 96);
            reg_fence_f(hm2);
            reg_fence_f(hm3);
            if (tail1) {
              mask_tail32(sr + 64, e1, 0, Nb, last_valid);
              mask_tail32(sr + 96, e1, 1, Nb, last_valid);
              mx1 = fmaxf(max32(sr + 64), max32(sr + 96));
            } else {
              mx1 = fmaxf(hm2, hm3);
            }
          }
        }
        // the factors are positive: the max commutes with them
        const float bmax = fmaxf(mx0 * c0, mx1 * c1);
        // the running max after step g - 1 (none before the tile's first step)
        float m_prev = -INFINITY;
        if (j > 0) {
          uint64_t hv;
          if (!wait_handoff(g - 1, hv)) {
            if (lane == 0) fail(kSiteHandoff);
            stop = true;
            break;
          }
          m_prev = __uint_as_float(static_cast<uint32_t>(hv));
        }
        float m_new = m_prev;
        if (bmax > m_prev + kRescaleLog2) m_new = bmax;  // also the first finite block
        *hand_mine = (static_cast<uint64_t>(static_cast<uint32_t>(g)) << 32) | __float_as_uint(m_new);
        const bool raised = (m_new != m_prev) && (m_prev != -INFINITY);
        if (__any_sync(full, raised)) {
          // O holds this tile's PVs of the steps before g; the last of them,
          // PV(g - 1), must be done before O is rescaled (PV(g) waits for this
          // step's p_full, so no later PV can be running). A parity wait needs
          // the barrier within one phase of the one waited for: S(g) is
          // written after PV(g - 3) in the tensor pipe's order, so on the
          // barrier of g - 1's parity the phase before it is done.
          if (!mbar_wait_warp(bar(L::bPVDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_sig)) {
            if (lane == 0) fail(kSitePVDone);
            stop = true;
            break;
          }
          tc_fence_after();
          const float alpha = raised ? fast_exp2(m_prev - m_new) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * cc, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(lane_base + kColO + 32 * cc, o);
          }
        }
        // P over the step's keys: 32 columns (two fp16 per column) per key
        // block at the start of the consumed S columns.
        float rs = 0.f;
        {
          uint32_t pk[32];
          if (mem0) {
            rs = exp_pack32(sr, c0, -m_new, pk);
            rs += exp_pack32(sr + 32, c0, -m_new, pk + 16);
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) pk[u] = 0u;
          }
          tmem_st32(lane_base + s_col, pk);
        }
        if (two) {
          uint32_t pk[32];
          if (mem1) {
            rs += exp_pack32(sr + 64, c1, -m_new, pk);
            rs += exp_pack32(sr + 96, c1, -m_new, pk + 16);
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) pk[u] = 0u;
          }
          tmem_st32(lane_base + s_col + 32, pk);
        }
        // this warpgroup's sum, carried to the new max
        l_run = (l_run > 0.f ? l_run * fast_exp2(m_run - m_new) : 0.f) + rs;
        m_run = m_new;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::bPFull + sb));
      }
      gs += n_steps;
      if (!stop) mbar_arrive(bar(L::bInfoEmpty + x));     // done with this walk

      // -------------------------------------------------------- epilogue
      // The two threads of the row add their partial sums (each carried to
      // the later max); each writes half of the output columns once every
      // PV of the tile is done.
      if (!stop) {
        stop = !mbar_wait_warp(bar(L::bTileDone), it & 1, abort_sig);
        if (stop && lane == 0) fail(kSiteFin);
      }
      float m_oth, l_oth;
      if (pair_xchg(m_run, l_run, stop, m_oth, l_oth)) break;
      tc_fence_after();
      // O is scaled to the tile's last max, the larger of the two
      const float m_tot = fmaxf(m_run, m_oth);
      const float f_own = l_run > 0.f ? fast_exp2(m_run - m_tot) : 0.f;
      const float f_oth = l_oth > 0.f ? fast_exp2(m_oth - m_tot) : 0.f;
      const float l_tot = l_run * f_own + l_oth * f_oth;
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const bool row_ok = qb >= 0 && t < S;
      const int c0 = sm * (D / 2);              // this thread's output columns
      uint16_t* orow = a.o + b * a.os[0] + static_cast<int64_t>(t) * a.os[1] + h * a.os[2] + c0;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + c0 + 32 * cc, ov);
        tmem_wait_ld();
        reg_fence32(ov);
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              // a row without weight may face an O this tile never wrote:
              // select, never multiply, so stale TMEM cannot leak in
              f[u] = l_tot > 0.f ? __uint_as_float(ov[8 * v + u]) * inv_l : 0.f;
            }
            uint4 wv;
            wv.x = pack_bf162(f[0], f[1]);
            wv.y = pack_bf162(f[2], f[3]);
            wv.z = pack_bf162(f[4], f[5]);
            wv.w = pack_bf162(f[6], f[7]);
            *reinterpret_cast<uint4*>(orow + 32 * cc + 8 * v) = wv;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::bOFree));             // O read
      if (row_ok && sm == 0 && a.lse) {
        const float lse = l_tot > 0.f ? m_tot * 0.69314718055994531f + logf(l_tot) : -INFINITY;
        a.lse[(static_cast<int64_t>(b) * a.H + h) * S + t] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// V [B,S,H,D] bf16 -> vt [B*H][D][s_pad] fp16 (key-contiguous). Each thread
// converts an 8-token x 8-d block: eight 16-byte loads (one token row each,
// the D/8 threads of a token group read whole rows), a transpose in
// registers, eight 16-byte stores (one d row each). Tokens in [S, s_pad)
// are written as zeros. grid (ceil(s_pad / tokens per CTA), H, B), 256 threads.
template <int D>
__global__ void __launch_bounds__(256)
pack_v_kernel(const uint16_t* __restrict__ v, int64_t vs0, int64_t vs1, int64_t vs2, int S, int H,
              int s_pad, uint16_t* __restrict__ vt, int32_t* dev_status) {
  constexpr int kChunks = D / 8;                     // threads per token group
  constexpr int kTokens = 256 / kChunks * 8;         // tokens per CTA
  const int c = threadIdx.x % kChunks, g = threadIdx.x / kChunks;
  const int h = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * kTokens + g * 8;
  bool range = false;
  if (t0 < s_pad) {
    uint4 w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      w[q] = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + q < S)
        w[q] = __ldg(reinterpret_cast<const uint4*>(v + b * vs0 + static_cast<int64_t>(t0 + q) * vs1 +
                                                    h * vs2 + 8 * c));
    }
    uint16_t* dst = vt + (static_cast<int64_t>(b) * H + h) * D * s_pad + static_cast<int64_t>(8 * c) * s_pad + t0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      float f[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t word = (&w[q].x)[p >> 1];
        f[q] = __uint_as_float((p & 1) ? (word & 0xffff0000u) : (word << 16));
        range |= fabsf(f[q]) > 65504.f && !isinf(f[q]);
      }
      uint4 o;
      o.x = pack_half2(f[0], f[1]);
      o.y = pack_half2(f[2], f[3]);
      o.z = pack_half2(f[4], f[5]);
      o.w = pack_half2(f[6], f[7]);
      *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(p) * s_pad) = o;
    }
  }
  if (__syncthreads_or(range) && threadIdx.x == 0) set_status(dev_status, SA_DEV_RANGE);
}

template <int D, bool kF8>
cudaError_t launch_attn_d(const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  constexpr int smem = Smem<D, kF8>::kBytes;
  static_assert(smem <= 227 * 1024, "attention tile does not fit shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kF8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.n_tiles < sms ? a.n_tiles : sms;   // persistent: one CTA per SM
  attn_fwd_kernel<D, kF8><<<grid, kThreads, smem, st>>>(m.q, m.k, m.vt, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_v(const uint16_t* v, const int64_t vs[3], int B, int S, int H, int D,
                          int s_pad, uint16_t* vt, int32_t* dev_status, cudaStream_t st) {
  const int per_cta = 256 / (D / 8) * 8;
  dim3 grid((s_pad + per_cta - 1) / per_cta, H, B);
  if (D == 128)
    pack_v_kernel<128><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], S, H, s_pad, vt, dev_status);
  else
    pack_v_kernel<64><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], S, H, s_pad, vt, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_attn(int D, const AttnMaps& m, const AttnArgs& a, cudaStream_t st) {
  if (a.q_exp != nullptr) return launch_attn_d<128, true>(m, a, st);   // 8-bit scores: D = 128
  return D == 128 ? launch_attn_d<128, false>(m, a, st) : launch_attn_d<64, false>(m, a, st);
}

}  // namespace sa
