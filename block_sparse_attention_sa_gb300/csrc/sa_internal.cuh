// sa_internal.cuh -- shared between the C-ABI host code and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sa.h"

namespace sa {

constexpr int kBlock = 64;          // query/key block (tokens)
constexpr int kMaxNbAttn = 4096;    // key blocks the attention tile can list
constexpr int kScoreTile = 64;      // pooled-score tile (query blocks x key blocks)

inline int num_blocks(int S) { return (S + kBlock - 1) / kBlock; }

// ------------------------------------------------------------ routing ---

struct RouteLayout {      // byte offsets into the caller's route workspace
  size_t qbar32, kbar32, qbar64, kbar64, qnorm, knorm, kmax;
  size_t part_m, part_s, scores, bits, counts, nflag, flags, total;
  int Nb, n_ct, words;
  int Nq, n_qt;           // query blocks per head and their score tiles
  int64_t rows;           // CSR rows, B*H*Nb (one per 64-token query block)
  int64_t qrows;          // routed rows, B*H*Nq (one per query block)
};

// Query block size of a route: sa_params.q_block, 0 meaning 64.
inline int q_block_of(const sa_params& p) { return p.q_block == 0 ? kBlock : p.q_block; }

RouteLayout route_layout(const sa_params& p);

struct RouteArgs {
  const uint16_t* q;      // bf16 bits
  const uint16_t* k;
  int64_t qs[3], ks[3];   // element strides of b, s, h
  int B, S, H, D, Nb, n_ct, words, n_sink;
  int qblk, qr, Nq;       // query block (64 or 128), qblk / 64, query blocks per head
  int n_prefix_q;         // query blocks meeting the prefix, ceil(P / qblk)
  float scale;            // fp32 softmax scale
  double scale64;         // fp64 softmax scale
  float log_tau_over_nb;  // logf(tau) - logf(Nb)  (tau > 0)
  double tau_over_nb;     // tau / Nb in fp64
  int keep_all;           // tau == 0 outside SA_ROUTE_TOP_MASS
  int mode;               // SA_ROUTE_*
  float tau;              // top-mass: the mass to reach
  double tau64;
  float gamma;            // fp32 dot-product error constant
  char* ws;
  RouteLayout L;
  int32_t* row_ptr;
  int32_t* col_idx;
  int64_t col_cap;
  int32_t* dev_status;
};

// QK-norm + RoPE prologue (sa_qk_prologue): reads RouteArgs::q, k.
struct PrologueArgs {
  const float* gamma_q;    // [D] or nullptr (ones)
  const float* gamma_k;
  const float* cos;        // [S][D/2] or nullptr (no rotation; then sin too)
  const float* sin;
  float eps;
  uint16_t* q_out;         // bf16 bits, strides of q (may equal q)
  uint16_t* k_out;         // strides of k (may equal k)
};

cudaError_t launch_route(const RouteArgs& a, cudaStream_t st);   // pool + select
// pa == nullptr: pool q, k; else the prologue writes q_out, k_out and pools them
cudaError_t launch_pool(const RouteArgs& a, const PrologueArgs* pa, cudaStream_t st);
cudaError_t launch_route_select(const RouteArgs& a, cudaStream_t st);

// ---------------------------------------------------------- attention ---

// ---------------------------------------------------- tile pairing ---

constexpr int kPairWindow = 32;     // query blocks pair only with blocks this close

struct PairArgs {
  const int32_t* row_ptr;  // the route (CSR)
  const int32_t* col_idx;
  int16_t* cand;           // [B*H*Nb][2 kPairWindow] candidates of each block, best first
  uint32_t* pairs;         // [B*H][n_pairs] a | b << 16 (a < b; b = 0xffff: a alone)
  int64_t nnz_row;         // B*H*Nb: row_ptr[nnz_row] is the route's entry count
  int Nb, n_pairs;
};

size_t pair_cand_bytes(int64_t rows);
cudaError_t launch_pair(const PairArgs& a, int BH, cudaStream_t st);

struct AttnArgs {
  const int32_t* row_ptr;  // nullptr: dense (every key block)
  const int32_t* col_idx;
  const uint32_t* pairs;   // tile list from launch_pair; nullptr: blocks (2p, 2p+1)
  uint16_t* o;             // bf16 bits
  float* lse;
  int32_t* dev_status;
  int64_t os[3];
  int B, S, H, Nb, n_pairs;
  float scale_log2;        // softmax_scale * log2(e)
  int* tile_counter;       // zeroed before the launch; tiles are taken in order
  int* grid_abort;         // zeroed before the launch; set by a CTA whose wait gave up
  int64_t nnz_row;         // B*H*Nb: row_ptr[nnz_row] is the route's entry count
  int n_tiles;             // B * H * n_pairs
  const int8_t* q_exp;     // 8-bit scores: [B*H*Nb] scale exponents (nullptr: bf16)
  const int8_t* k_exp;
};

struct AttnMaps {
  CUtensorMap q, k, vt;    // q, k: bf16, or the e4m3 codes for 8-bit scores
};

// 8-bit (e4m3) copies of Q and K with one power-of-two scale exponent per
// (batch, head, 64-token block); D = 128.
struct QuantArgs {
  const uint16_t* q;       // bf16 bits
  const uint16_t* k;
  int64_t qs[3], ks[3];    // element strides of b, s, h
  uint8_t* q8;             // e4m3 codes, [B, S, H, D] with strides y_stride (bytes)
  uint8_t* k8;
  int64_t y_stride[3];
  int8_t* q_exp;           // [B*H*Nb] scale exponents
  int8_t* k_exp;
  int B, S, H, Nb;
  int32_t* dev_status;
};

cudaError_t launch_quant(const QuantArgs& a, cudaStream_t st);

// Repacks V [B,S,H,D] bf16 into vt [B*H][D][s_pad] fp16 (key-contiguous).
cudaError_t launch_pack_v(const uint16_t* v, const int64_t vs[3], int B, int S, int H, int D,
                          int s_pad, uint16_t* vt, int32_t* dev_status, cudaStream_t st);

cudaError_t launch_attn(int D, const AttnMaps& maps, const AttnArgs& a, cudaStream_t st);

}  // namespace sa
