// pair.cu -- chooses which two query blocks of a head share a 128-row
// attention tile.
//
// The attention tile is 128 query rows (tcgen05 M = 128) while the route is
// per 64-row query block, so every tile holds two query blocks a and b and
// walks the union of their key lists; a key block listed by only one of them
// is still multiplied for all 128 rows and masked for the other half. A head
// therefore costs sum over its tiles of ceil(|R_a u R_b| / 2) steps of 128
// keys, and because |R_a u R_b| = |R_a| + |R_b| - |R_a n R_b|, the pairing
// with the least work is the perfect matching of the head's query blocks
// with the largest summed intersection. Pairing neighbours (2p, 2p+1) is
// exact only where neighbours route alike; on a 3-D latent grid laid out
// frame after frame, the block with the most similar key list is often the
// same spatial patch one frame away.
//
// The matching taken is the greedy one (heaviest edge first) over the
// candidates within kPairWindow blocks of each other, computed as a locally
// dominant matching: every unmatched block points at its heaviest unmatched
// candidate and mutual pointers pair up, round after round. With a strict
// total order on the edges this is exactly the greedy matching, and the
// heaviest remaining edge is always mutual, so every round pairs at least
// one couple. Blocks left without a candidate pair up in index order.
// Edge order: intersection; then the neighbour pair (2p, 2p+1), so that a
// route where every list is alike (e.g. every block kept) gives the
// neighbour pairing in one round; then a fixed hash of the edge, so that
// runs of equal weights do not resolve one pair per round as an index order
// would; the edge's own (lo, d) in the low bits make every key distinct.
//
// Kernels, in launch order:
//   pair_rank   per (head, 64-row chunk), across all SMs: bitmaps of the rows
//               within kPairWindow of the chunk, built from the CSR in shared
//               memory; for every block of the chunk the keys of its 2W
//               candidates (intersections by popcount), sorted by a warp
//               bitonic network; writes the candidates in key order, int16
//               [B*H*Nb][2W] (-1 past the valid ones).
//   pair_match  one CTA per head: the rounds above on the head's lists in
//               shared memory, where a block whose choice was taken steps
//               along its sorted list to the next unmatched candidate; writes the tile list [B*H][ceil(Nb/2)]
//               of (a | b << 16), a < b, b = 0xffff for the odd block alone,
//               ordered by a.
#include "sa_internal.cuh"

namespace sa {

namespace {

constexpr int kW = kPairWindow;        // candidates: blocks within kW of a block
constexpr int kCand = 2 * kW;          // two per lane
static_assert(kCand == 64, "the bitonic network below sorts two keys per lane");
constexpr int kChunk = 64;             // blocks ranked per pair_rank CTA
constexpr int kRankThreads = 512;
constexpr int kMaxRows = kChunk + 2 * kW;   // bitmap rows a pair_rank CTA holds
constexpr int kMatchThreads = 512;
constexpr uint32_t kNoPartner = 0xffffu;
constexpr unsigned kFull = 0xffffffffu;

// Bitmap row stride in words: whole 16-byte groups (vector loads), an odd
// number of them, so eight consecutive rows hit eight different bank groups.
__host__ __device__ inline int bitmap_stride(int words) {
  const int g = (words + 3) >> 2;
  return 4 * (g | 1);
}

__device__ __forceinline__ uint32_t edge_hash(uint32_t x) {
  x *= 0x9e3779b1u;
  x ^= x >> 15;
  x *= 0x2c1b3c6du;
  x ^= x >> 12;
  return x;
}

// Key of edge (lo, lo + d) with weight w; 0 is below every edge's key.
__device__ __forceinline__ uint64_t edge_key(uint32_t w, int lo, int d) {
  const uint64_t natural = (d == 1 && (lo & 1) == 0) ? 1u : 0u;
  const uint64_t hsh = edge_hash(static_cast<uint32_t>(lo * 128 + d)) >> 8;   // 24 bits
  return (static_cast<uint64_t>(w) << 44) | (natural << 43) | (hsh << 19) |
         (static_cast<uint64_t>(d) << 12) | static_cast<uint64_t>(lo);
}

// One CSR row -> bitmap (whole warp), for the slow path: rows that break the
// CSR contract count as empty (the attention planner reports them) and
// entries outside [0, Nb) are skipped.
__device__ void row_bits_checked(const int32_t* row_ptr, const int32_t* col_idx, int64_t r,
                                 int Nb, int nnz, uint32_t* bits, int lane) {
  const int beg = row_ptr[r], end = row_ptr[r + 1];
  if (beg < 0 || end < beg || end - beg > Nb || end > nnz) return;
  for (int e = beg + lane; e < end; e += 32) {
    const int j = col_idx[e];
    if (j >= 0 && j < Nb) atomicOr(&bits[j >> 5], 1u << (j & 31));
  }
}

// grid (ceil(Nb / 64), B*H), 512 threads; dynamic smem: row_ptr slice
// [kMaxRows + 1] ints, then bitmaps [kMaxRows][ld].
__global__ void __launch_bounds__(kRankThreads) pair_rank_kernel(PairArgs a) {
  extern __shared__ uint32_t sm[];
  const int bh = blockIdx.y, a0 = blockIdx.x * kChunk;
  const int Nb = a.Nb, words = (Nb + 31) >> 5, ld = bitmap_stride(words);
  const int r_lo = max(0, a0 - kW), r_hi = min(Nb, a0 + kChunk + kW);
  const int rows = r_hi - r_lo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* rp = reinterpret_cast<int*>(sm);
  uint32_t* bits = sm + kMaxRows + 4;
  const int64_t row0 = static_cast<int64_t>(bh) * Nb + r_lo;
  for (int i = threadIdx.x; i <= rows; i += kRankThreads) rp[i] = a.row_ptr[row0 + i];
  for (int i = threadIdx.x; i < rows * ld; i += kRankThreads) bits[i] = 0u;
  __syncthreads();
  const int nnz = a.row_ptr[a.nnz_row];   // entries of the whole route
  bool valid = rp[0] >= 0 && rp[rows] <= nnz;
  for (int i = threadIdx.x; i < rows; i += kRankThreads)
    valid = valid && rp[i + 1] >= rp[i] && rp[i + 1] - rp[i] <= Nb;
  if (__syncthreads_and(valid)) {
    // The rows' entries are one contiguous range of col_idx: coalesced loads,
    // eight in flight per thread; a thread's entries ascend, so its row
    // cursor only moves forward.
    const int64_t e_beg = rp[0], e_end = rp[rows];
    int row = 0;
    for (int64_t e0 = e_beg + threadIdx.x; e0 < e_end; e0 += 8 * kRankThreads) {
      int j[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t e = e0 + q * kRankThreads;
        j[q] = e < e_end ? __ldg(a.col_idx + e) : -1;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t e = e0 + q * kRankThreads;
        if (e >= e_end) break;
        while (rp[row + 1] <= e) ++row;
        if (j[q] >= 0 && j[q] < Nb) atomicOr(&bits[row * ld + (j[q] >> 5)], 1u << (j[q] & 31));
      }
    }
  } else {
    for (int i = warp; i < rows; i += kRankThreads / 32)
      row_bits_checked(a.row_ptr, a.col_idx, row0 + i, Nb, nnz, bits + i * ld, lane);
  }
  __syncthreads();

  for (int i = warp; i < kChunk; i += kRankThreads / 32) {
    const int u = a0 + i;
    if (u >= Nb) break;
    const uint4* bu = reinterpret_cast<const uint4*>(bits + (u - r_lo) * ld);
    uint64_t k[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      // lane l holds blocks u - kW + l and u + 1 + l: every block within kW but u
      const int v = s == 0 ? u - kW + lane : u + 1 + lane;
      k[s] = 0;
      if (v >= 0 && v < Nb) {
        const uint4* bv = reinterpret_cast<const uint4*>(bits + (v - r_lo) * ld);
        int c0 = 0, c1 = 0;
        for (int g = 0; g < ld / 4; ++g) {
          const uint4 x = bu[g], y = bv[g];
          c0 += __popc(x.x & y.x) + __popc(x.y & y.y);
          c1 += __popc(x.z & y.z) + __popc(x.w & y.w);
        }
        k[s] = edge_key(static_cast<uint32_t>(c0 + c1), min(u, v), abs(u - v));
      }
    }
    // bitonic sort of the 64 keys, descending (key k[s] of lane l is element 2 l + s)
#pragma unroll
    for (int size = 2; size <= kCand; size <<= 1) {
      const bool desc = ((2 * lane) & size) == 0;
#pragma unroll
      for (int stride = size >> 1; stride >= 2; stride >>= 1) {
        const bool lower = ((2 * lane) & stride) == 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint64_t o = __shfl_xor_sync(kFull, k[s], stride >> 1);
          k[s] = (lower == desc) ? (k[s] > o ? k[s] : o) : (k[s] < o ? k[s] : o);
        }
      }
      if ((k[0] < k[1]) == desc) {
        const uint64_t t = k[0];
        k[0] = k[1];
        k[1] = t;
      }
    }
    uint32_t out[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int lo = static_cast<int>(k[s] & 4095u), d = static_cast<int>((k[s] >> 12) & 127u);
      out[s] = k[s] == 0 ? 0xffffu : static_cast<uint32_t>(lo == u ? u + d : lo);
    }
    reinterpret_cast<uint32_t*>(a.cand + (static_cast<int64_t>(bh) * Nb + u) * kCand)[lane] =
        out[0] | (out[1] << 16);
  }
}

// Exclusive prefix sum over the block (kMatchThreads threads); also returns the total.
__device__ int block_excl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < kMatchThreads / 32 ? warp_tot[lane] : 0;
    int si = s;
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(kFull, si, off);
      if (lane >= off) si += t;
    }
    warp_tot[lane] = si - s;        // exclusive over warps
    if (lane == 31) warp_tot[32] = si;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  total = warp_tot[32];
  __syncthreads();                  // warp_tot is reused by the next scan
  return r;
}

// Candidates per block that pair_match keeps in shared memory (the rest of
// a list is read from global memory): all 2W while they fit, else a prefix
// that is a multiple of 8.
__host__ __device__ inline int match_prefix(int Nb) {
  const int t = (200 * 1024 - 8 * Nb) / (2 * Nb) - 8;
  return t >= kCand ? kCand : (t < 8 ? 8 : t & ~7);
}

// Row stride of the lists in shared memory (int16): the prefix plus 8, so
// consecutive blocks' lists start in different banks.
__host__ __device__ inline int match_stride(int Nb) { return match_prefix(Nb) + 8; }

__host__ __device__ inline size_t match_smem(int Nb) {
  return static_cast<size_t>(Nb) * match_stride(Nb) * 2 + 8 * static_cast<size_t>(Nb) + 16;
}

// grid (B*H), kMatchThreads threads; dynamic smem: the head's sorted lists
// (their first match_prefix(Nb) entries, rows match_stride(Nb) apart), then
// mate, best, pos, order (int16 [Nb] each).
__global__ void __launch_bounds__(kMatchThreads) pair_match_kernel(PairArgs a) {
  extern __shared__ __align__(16) int16_t smem_m[];
  __shared__ int warp_tot[33];
  __shared__ int n_need;
  const int bh = blockIdx.x, Nb = a.Nb, T = match_prefix(Nb), TS = match_stride(Nb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int16_t* lists = smem_m;
  int16_t* mate = lists + static_cast<size_t>(Nb) * TS;
  int16_t* best = mate + Nb;       // -1: not chosen yet, -2: no candidate left
  int16_t* pos = best + Nb;        // place of best[u] in u's sorted list
  int16_t* order = pos + Nb;
  const int16_t* cand = a.cand + static_cast<int64_t>(bh) * Nb * kCand;
  {
    const int vec = T / 8;         // 16-byte pieces of a list prefix
    for (int i = threadIdx.x; i < Nb * vec; i += kMatchThreads) {
      const int u = i / vec, c = i % vec;
      reinterpret_cast<uint4*>(lists + static_cast<size_t>(u) * TS)[c] =
          __ldg(reinterpret_cast<const uint4*>(cand + static_cast<size_t>(u) * kCand) + c);
    }
  }
  for (int i = threadIdx.x; i < Nb; i += kMatchThreads) {
    mate[i] = -1;
    best[i] = -1;
    pos[i] = -1;
  }
  auto entry = [&](int u, int p) -> int {
    return p < T ? lists[u * TS + p] : cand[static_cast<int64_t>(u) * kCand + p];
  };
  __syncthreads();

  for (int round = 0; round <= Nb; ++round) {
    // An unmatched block whose choice is unset or was taken chooses the first
    // candidate still unmatched after its old choice in its sorted list: the
    // ones before are matched for good, so that one is its heaviest
    // unmatched candidate. The next entry is checked here; a block whose next
    // entry is taken too is queued for a whole-warp scan.
    if (threadIdx.x == 0) n_need = 0;
    __syncthreads();
    for (int u = threadIdx.x; u < Nb; u += kMatchThreads) {
      const int bu = best[u];
      if (mate[u] >= 0 || bu == -2 || (bu >= 0 && mate[bu] < 0)) continue;
      const int p = pos[u] + 1;
      const int v = p < kCand ? entry(u, p) : -1;
      if (v < 0) {
        best[u] = -2;
      } else if (mate[v] < 0) {
        best[u] = static_cast<int16_t>(v);
        pos[u] = static_cast<int16_t>(p);
      } else {
        pos[u] = static_cast<int16_t>(p);
        order[atomicAdd(&n_need, 1)] = static_cast<int16_t>(u);
      }
    }
    __syncthreads();
    const int nn = n_need;
    for (int x = warp; x < nn; x += kMatchThreads / 32) {
      const int u = order[x];
      int pick = -2, at = kCand;
      for (int p0 = pos[u] + 1; p0 < kCand; p0 += 32) {
        const int p = p0 + lane;
        const int v = p < kCand ? entry(u, p) : -1;
        const bool end = p >= kCand || v < 0;
        const bool free = !end && mate[v] < 0;
        const unsigned fb = __ballot_sync(kFull, free), eb = __ballot_sync(kFull, end);
        const unsigned first = fb & (eb ? ((eb & (0u - eb)) - 1u) : kFull);  // before any end
        if (first) {
          const int l = __ffs(first) - 1;
          pick = __shfl_sync(kFull, v, l);
          at = p0 + l;
          break;
        }
        if (eb) break;
      }
      if (lane == 0) {
        best[u] = static_cast<int16_t>(pick);
        pos[u] = static_cast<int16_t>(at < kCand ? at : kCand - 1);
      }
    }
    __syncthreads();
    // mutual choices pair up (the heaviest remaining edge always is mutual)
    int any = 0;
    for (int u = threadIdx.x; u < Nb; u += kMatchThreads) {
      const int v = best[u];
      if (mate[u] < 0 && v > u && best[v] == u) {
        mate[u] = static_cast<int16_t>(v);
        mate[v] = static_cast<int16_t>(u);
        any = 1;
      }
    }
    if (!__syncthreads_or(any)) break;
  }

  const int per = (Nb + kMatchThreads - 1) / kMatchThreads;
  const int v0 = threadIdx.x * per, v1 = min(Nb, v0 + per);
  // blocks without a candidate: pair them in index order
  int mine = 0;
  for (int u = v0; u < v1; ++u) mine += mate[u] < 0;
  int total = 0;
  int rank = block_excl_scan(mine, warp_tot, total);
  for (int u = v0; u < v1; ++u)
    if (mate[u] < 0) order[rank++] = static_cast<int16_t>(u);
  __syncthreads();
  for (int k = threadIdx.x; 2 * k + 1 < total; k += kMatchThreads) {
    const int u = order[2 * k], v = order[2 * k + 1];
    mate[u] = static_cast<int16_t>(v);
    mate[v] = static_cast<int16_t>(u);
  }
  __syncthreads();

  // one tile per pair (and one for a block left alone), ordered by its lower block
  int lead = 0;
  for (int u = v0; u < v1; ++u) lead += (mate[u] < 0 || u < mate[u]);
  int slot = block_excl_scan(lead, warp_tot, total);
  uint32_t* out = a.pairs + static_cast<int64_t>(bh) * a.n_pairs;
  for (int u = v0; u < v1; ++u) {
    const int m = mate[u];
    if (m >= 0 && m < u) continue;
    if (slot < a.n_pairs) out[slot] = static_cast<uint32_t>(u) | ((m < 0 ? kNoPartner : m) << 16);
    ++slot;
  }
}

}  // namespace

size_t pair_cand_bytes(int64_t rows) { return static_cast<size_t>(rows) * kCand * sizeof(int16_t); }

cudaError_t launch_pair(const PairArgs& a, int BH, cudaStream_t st) {
  const int words = (a.Nb + 31) >> 5;
  const size_t smem_r = (kMaxRows + 4 + static_cast<size_t>(kMaxRows) * bitmap_stride(words)) * 4;
  cudaError_t e = cudaFuncSetAttribute(pair_rank_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_r));
  if (e != cudaSuccess) return e;
  pair_rank_kernel<<<dim3((a.Nb + kChunk - 1) / kChunk, BH), kRankThreads, smem_r, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smem_m = match_smem(a.Nb);
  e = cudaFuncSetAttribute(pair_match_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_m));
  if (e != cudaSuccess) return e;
  pair_match_kernel<<<BH, kMatchThreads, smem_m, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
