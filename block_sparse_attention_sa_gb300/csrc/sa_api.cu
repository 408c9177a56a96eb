// sa_api.cu -- the extern "C" boundary: argument checks, workspace layout,
// TMA descriptor encoding and the launch sequence of each entry point.
#include <cmath>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "sa_internal.cuh"

namespace sa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool strides_ok(const int64_t s[3]) {
  for (int i = 0; i < 3; ++i)
    if (s[i] <= 0 || (s[i] & 7) != 0) return false;
  return true;
}

sa_status check_params(const sa_params* p) {
  if (!p) return SA_ERR_INVALID_ARG;
  if (p->B < 1 || p->S < 1 || p->H < 1 || p->block != kBlock) return SA_ERR_INVALID_ARG;
  if (p->prefix_len < 0 || p->prefix_len > p->S) return SA_ERR_INVALID_ARG;
  if (!(p->tau >= 0.f) || !std::isfinite(p->tau)) return SA_ERR_INVALID_ARG;
  if (!(p->softmax_scale >= 0.f) || !std::isfinite(p->softmax_scale)) return SA_ERR_INVALID_ARG;
  if (p->route_mode < SA_ROUTE_THRESHOLD || p->route_mode > SA_ROUTE_TOP_MASS)
    return SA_ERR_INVALID_ARG;
  if (p->q_block != 0 && p->q_block != kBlock && p->q_block != 2 * kBlock) return SA_ERR_INVALID_ARG;
  if (p->route_mode == SA_ROUTE_TOP_MASS && p->tau > 1.f) return SA_ERR_INVALID_ARG;
  if (p->qk_format != SA_QK_BF16 && p->qk_format != SA_QK_FP8) return SA_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return p->D > 0 ? SA_ERR_UNSUPPORTED : SA_ERR_INVALID_ARG;
  if (p->qk_format == SA_QK_FP8 && p->D != 128) return SA_ERR_UNSUPPORTED;
  if (p->H > 65535 || p->B > 65535) return SA_ERR_UNSUPPORTED;
  const int64_t nb = num_blocks(p->S);
  const int64_t max_nnz = static_cast<int64_t>(p->B) * p->H * nb * nb;
  if (max_nnz > INT32_MAX) return SA_ERR_UNSUPPORTED;  // row_ptr is int32
  return SA_OK;
}

double scale64_of(const sa_params* p) {
  return p->softmax_scale > 0.f ? static_cast<double>(p->softmax_scale)
                                : 1.0 / std::sqrt(static_cast<double>(p->D));
}

sa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SA_OK : SA_ERR_CUDA; }

int s_pad_of(int S) { return (S + 7) & ~7; }

// [B, S, H, D] bf16 -> 4-D map (D, S, H, B), box 64 x 64, 128-byte swizzle.
sa_status encode_bshd(CUtensorMap* m, const void* base, const sa_params* p, const int64_t st[3]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SA_ERR_CUDA;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->D), static_cast<cuuint64_t>(p->S),
                              static_cast<cuuint64_t>(p->H), static_cast<cuuint64_t>(p->B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[1]) * 2,
                                 static_cast<cuuint64_t>(st[2]) * 2,
                                 static_cast<cuuint64_t>(st[0]) * 2};
  const cuuint32_t box[4] = {64, 64, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_INVALID_ARG;
}

// vt [B*H][D][s_pad] fp16 -> 3-D map (S, D, B*H), box 64 keys x D rows.
sa_status encode_vt(CUtensorMap* m, const void* base, const sa_params* p) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SA_ERR_CUDA;
  const cuuint64_t sp = static_cast<cuuint64_t>(s_pad_of(p->S));
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->S), static_cast<cuuint64_t>(p->D),
                              static_cast<cuuint64_t>(p->B) * p->H};
  const cuuint64_t strides[2] = {sp * 2, sp * 2 * static_cast<cuuint64_t>(p->D)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(p->D), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_INVALID_ARG;
}

size_t vt_bytes(const sa_params* p) {
  return static_cast<size_t>(p->B) * p->H * p->D * s_pad_of(p->S) * 2;
}

// e4m3 codes [B, S, H, D], contiguous -> 4-D map (D, S, H, B), box 128 x 64
// (one 128-byte row per token), 128-byte swizzle.
sa_status encode_bshd_u8(CUtensorMap* m, const void* base, const sa_params* p) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SA_ERR_CUDA;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->D), static_cast<cuuint64_t>(p->S),
                              static_cast<cuuint64_t>(p->H), static_cast<cuuint64_t>(p->B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p->H) * p->D,
                                 static_cast<cuuint64_t>(p->D),
                                 static_cast<cuuint64_t>(p->S) * p->H * p->D};
  const cuuint32_t box[4] = {128, 64, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_INVALID_ARG;
}

size_t codes_bytes(const sa_params* p) {
  return static_cast<size_t>(p->B) * p->S * p->H * p->D;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Attention workspace, each part 256-byte aligned: V repacked to fp16, the
// persistent kernel's tile counter, the pairing's candidate lists, with
// 8-bit scores the e4m3 codes of Q and K and their scale exponents, and the
// tile list (last).
struct AttnLayout {
  size_t vt, counter, cand, q8, k8, qexp, kexp, pairs, total;
};

AttnLayout attn_layout(const sa_params* p) {
  const int Nb = num_blocks(p->S);
  const int64_t bh = static_cast<int64_t>(p->B) * p->H;
  AttnLayout L{};
  L.vt = 0;
  L.counter = align256(vt_bytes(p));
  L.cand = L.counter + 256;
  L.q8 = L.cand + align256(pair_cand_bytes(bh * Nb));
  const bool f8 = p->qk_format == SA_QK_FP8;
  L.k8 = L.q8 + (f8 ? align256(codes_bytes(p)) : 0);
  L.qexp = L.k8 + (f8 ? align256(codes_bytes(p)) : 0);
  L.kexp = L.qexp + (f8 ? align256(static_cast<size_t>(bh) * Nb) : 0);
  L.pairs = L.kexp + (f8 ? align256(static_cast<size_t>(bh) * Nb) : 0);
  L.total = L.pairs + align256(static_cast<size_t>(bh) * ((Nb + 1) / 2) * sizeof(uint32_t));
  return L;
}

size_t attn_ws_bytes(const sa_params* p) { return attn_layout(p).total; }

// The launch-time checks of the attention calls (q, k, o unchecked when
// null_qko_ok: sa_attn_prepare does not take them).
sa_status attn_check(const sa_params* p, const void* q, const void* k, const void* v,
                     const int32_t* row_ptr, const int32_t* col_idx, const void* o,
                     const void* ws, size_t ws_bytes, bool dense, bool need_v, bool need_qko) {
  const sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!ws || (need_v && !v) || (need_qko && (!q || !k || !o))) return SA_ERR_INVALID_ARG;
  if (!dense && (!row_ptr || !col_idx)) return SA_ERR_INVALID_ARG;
  if ((need_v && !aligned16(v)) || (need_qko && (!aligned16(q) || !aligned16(k) || !aligned16(o))))
    return SA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SA_ERR_INVALID_ARG;
  if (!strides_ok(p->q_stride) || !strides_ok(p->k_stride) || !strides_ok(p->v_stride) ||
      !strides_ok(p->o_stride))
    return SA_ERR_INVALID_ARG;
  if (num_blocks(p->S) > kMaxNbAttn) return SA_ERR_UNSUPPORTED;
  if (ws_bytes < attn_ws_bytes(p)) return SA_ERR_CAPACITY;
  return SA_OK;
}

// Tiles of two 64-token query blocks are paired from the route; a route of
// 128-token query blocks gives both halves of each tile (2i, 2i + 1) the
// same list, so the neighbour tiles are then exact.
bool uses_pairing(const sa_params* p, bool dense) {
  return !dense && num_blocks(p->S) > 2 && q_block_of(*p) == kBlock;
}

// First half of an attention call: V repacked into the workspace, and the
// tile pairs chosen from the route.
sa_status attn_prepare_launch(const sa_params* p, const void* v, const int32_t* row_ptr,
                              const int32_t* col_idx, void* ws, int32_t* dev_status,
                              cudaStream_t st, bool dense) {
  if (launch_pack_v(static_cast<const uint16_t*>(v), p->v_stride, p->B, p->S, p->H, p->D,
                    s_pad_of(p->S), static_cast<uint16_t*>(ws), dev_status, st) != cudaSuccess)
    return SA_ERR_CUDA;
  if (uses_pairing(p, dense)) {
    const AttnLayout L = attn_layout(p);
    char* wsb = static_cast<char*>(ws);
    const int Nb = num_blocks(p->S);
    PairArgs pa{};
    pa.row_ptr = row_ptr;
    pa.col_idx = col_idx;
    pa.cand = reinterpret_cast<int16_t*>(wsb + L.cand);
    pa.pairs = reinterpret_cast<uint32_t*>(wsb + L.pairs);
    pa.Nb = Nb;
    pa.n_pairs = (Nb + 1) / 2;
    pa.nnz_row = static_cast<int64_t>(p->B) * p->H * Nb;
    if (launch_pair(pa, p->B * p->H, st) != cudaSuccess) return SA_ERR_CUDA;
  }
  return SA_OK;
}

// Second half: the attention kernel over the prepared workspace.
sa_status attn_run_launch(const sa_params* p, const void* q, const void* k,
                          const int32_t* row_ptr, const int32_t* col_idx, void* o, float* lse,
                          void* ws, int32_t* dev_status, cudaStream_t st, bool dense) {
  sa_status s;
  AttnMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const AttnLayout L = attn_layout(p);
  char* wsb = static_cast<char*>(ws);
  const int Nb = num_blocks(p->S);
  const bool f8 = p->qk_format == SA_QK_FP8;
  if (f8) {
    // 8-bit scores: Q and K quantised into the workspace first
    QuantArgs qa{};
    qa.q = static_cast<const uint16_t*>(q);
    qa.k = static_cast<const uint16_t*>(k);
    for (int i = 0; i < 3; ++i) {
      qa.qs[i] = p->q_stride[i];
      qa.ks[i] = p->k_stride[i];
    }
    qa.q8 = reinterpret_cast<uint8_t*>(wsb + L.q8);
    qa.k8 = reinterpret_cast<uint8_t*>(wsb + L.k8);
    qa.y_stride[0] = static_cast<int64_t>(p->S) * p->H * p->D;
    qa.y_stride[1] = static_cast<int64_t>(p->H) * p->D;
    qa.y_stride[2] = p->D;
    qa.q_exp = reinterpret_cast<int8_t*>(wsb + L.qexp);
    qa.k_exp = reinterpret_cast<int8_t*>(wsb + L.kexp);
    qa.B = p->B;
    qa.S = p->S;
    qa.H = p->H;
    qa.Nb = Nb;
    qa.dev_status = dev_status;
    if (launch_quant(qa, st) != cudaSuccess) return SA_ERR_CUDA;
    if ((s = encode_bshd_u8(&maps.q, wsb + L.q8, p)) != SA_OK) return s;
    if ((s = encode_bshd_u8(&maps.k, wsb + L.k8, p)) != SA_OK) return s;
  } else {
    if ((s = encode_bshd(&maps.q, q, p, p->q_stride)) != SA_OK) return s;
    if ((s = encode_bshd(&maps.k, k, p, p->k_stride)) != SA_OK) return s;
  }
  if ((s = encode_vt(&maps.vt, ws, p)) != SA_OK) return s;
  AttnArgs a{};
  a.row_ptr = dense ? nullptr : row_ptr;
  a.col_idx = dense ? nullptr : col_idx;
  a.pairs = uses_pairing(p, dense) ? reinterpret_cast<uint32_t*>(wsb + L.pairs) : nullptr;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.dev_status = dev_status;
  for (int i = 0; i < 3; ++i) a.os[i] = p->o_stride[i];
  a.B = p->B;
  a.S = p->S;
  a.H = p->H;
  a.Nb = Nb;
  a.n_pairs = (Nb + 1) / 2;
  a.scale_log2 = static_cast<float>(scale64_of(p) * 1.4426950408889634);
  a.n_tiles = p->B * p->H * a.n_pairs;
  a.nnz_row = static_cast<int64_t>(p->B) * p->H * Nb;
  // the tile counter and the launch's abort word, zeroed together
  a.tile_counter = reinterpret_cast<int*>(wsb + L.counter);
  a.grid_abort = a.tile_counter + 1;
  a.q_exp = f8 ? reinterpret_cast<const int8_t*>(wsb + L.qexp) : nullptr;
  a.k_exp = f8 ? reinterpret_cast<const int8_t*>(wsb + L.kexp) : nullptr;
  if (cudaMemsetAsync(a.tile_counter, 0, 2 * sizeof(int), st) != cudaSuccess) return SA_ERR_CUDA;
  return from_cuda(launch_attn(p->D, maps, a, st));
}

sa_status attn_common(const sa_params* p, const void* q, const void* k, const void* v,
                      const int32_t* row_ptr, const int32_t* col_idx, void* o, float* lse,
                      void* ws, size_t ws_bytes, int32_t* dev_status, void* stream, bool dense) {
  sa_status s = attn_check(p, q, k, v, row_ptr, col_idx, o, ws, ws_bytes, dense, true, true);
  if (s != SA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = attn_prepare_launch(p, v, row_ptr, col_idx, ws, dev_status, st, dense)) != SA_OK)
    return s;
  return attn_run_launch(p, q, k, row_ptr, col_idx, o, lse, ws, dev_status, st, dense);
}

// sa_forward_host's copy streams and events, created on first use on each
// device and kept until the process exits.
constexpr int kHostGroups = 8;
struct HostPipe {
  std::mutex mu;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, in[kHostGroups] = {}, done[kHostGroups] = {};
  bool ok = false;
};

HostPipe* host_pipe(int dev) {
  constexpr int kMaxDevices = 64;
  static HostPipe pipes[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  HostPipe& hp = pipes[dev];
  std::call_once(once[dev], [&hp] {
    bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming) == cudaSuccess;
    for (int g = 0; ok && g < kHostGroups; ++g)
      ok = cudaEventCreateWithFlags(&hp.in[g], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.done[g], cudaEventDisableTiming) == cudaSuccess;
    hp.ok = ok;
  });
  return hp.ok ? &hp : nullptr;
}

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" {

void sa_params_init(sa_params* p, int32_t B, int32_t S, int32_t H, int32_t D, int32_t prefix_len,
                    float tau) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->B = B;
  p->S = S;
  p->H = H;
  p->D = D;
  p->block = kBlock;
  p->prefix_len = prefix_len;
  p->tau = tau;
  p->softmax_scale = 0.f;
  const int64_t st[3] = {static_cast<int64_t>(S) * H * D, static_cast<int64_t>(H) * D, D};
  for (int i = 0; i < 3; ++i) {
    p->q_stride[i] = st[i];
    p->k_stride[i] = st[i];
    p->v_stride[i] = st[i];
    p->o_stride[i] = st[i];
  }
}

int32_t sa_num_blocks(const sa_params* p) {
  return (p && p->S >= 1) ? num_blocks(p->S) : 0;
}

int64_t sa_route_rows(const sa_params* p) {
  if (check_params(p) != SA_OK) return 0;
  return static_cast<int64_t>(p->B) * p->H * num_blocks(p->S);
}

int64_t sa_route_max_nnz(const sa_params* p) {
  if (check_params(p) != SA_OK) return 0;
  const int64_t nb = num_blocks(p->S);
  return static_cast<int64_t>(p->B) * p->H * nb * nb;
}

size_t sa_route_workspace_bytes(const sa_params* p) {
  if (check_params(p) != SA_OK) return 0;
  return route_layout(*p).total;
}

size_t sa_attn_workspace_bytes(const sa_params* p) {
  if (check_params(p) != SA_OK) return 0;
  return attn_ws_bytes(p);
}

}  // extern "C"

namespace sa {
namespace {

// The router's launch arguments for p on the caller's workspace; q, k,
// row_ptr, col_idx are checked by the callers that use them.
sa_status route_args(const sa_params* p, const void* q, const void* k, int32_t* row_ptr,
                     int32_t* col_idx, int64_t col_cap, void* workspace, size_t ws_bytes,
                     int32_t* dev_status, RouteArgs* out) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!workspace || col_cap < 0) return SA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SA_ERR_INVALID_ARG;
  if (!strides_ok(p->q_stride) || !strides_ok(p->k_stride)) return SA_ERR_INVALID_ARG;
  const RouteLayout L = route_layout(*p);
  if (ws_bytes < L.total) return SA_ERR_CAPACITY;

  RouteArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  for (int i = 0; i < 3; ++i) {
    a.qs[i] = p->q_stride[i];
    a.ks[i] = p->k_stride[i];
  }
  a.B = p->B;
  a.S = p->S;
  a.H = p->H;
  a.D = p->D;
  a.Nb = L.Nb;
  a.n_ct = L.n_ct;
  a.words = L.words;
  a.n_sink = (p->prefix_len + kBlock - 1) / kBlock;
  a.qblk = q_block_of(*p);
  a.qr = a.qblk / kBlock;
  a.Nq = L.Nq;
  a.n_prefix_q = (p->prefix_len + a.qblk - 1) / a.qblk;
  a.scale64 = scale64_of(p);
  a.scale = static_cast<float>(a.scale64);
  a.mode = p->route_mode;
  a.tau = p->tau;
  a.tau64 = static_cast<double>(p->tau);
  a.keep_all = p->route_mode != SA_ROUTE_TOP_MASS && p->tau == 0.f;
  a.tau_over_nb = static_cast<double>(p->tau) / L.Nb;
  a.log_tau_over_nb = (a.keep_all || p->tau == 0.f) ? 0.f
                                 : static_cast<float>(std::log(static_cast<double>(p->tau)) -
                                                      std::log(static_cast<double>(L.Nb)));
  // gamma_n (1 + 1%) with u = 2^-24 and n = 16 + D/16 + 3: the score kernel
  // sums each dot product as 16-term FMA chains added into a running total,
  // after rounding qbar, kbar to fp32 and before scaling, so the fp32 score
  // error is at most gamma * scale * |qbar| |kbar| (Cauchy-Schwarz).
  const double u = std::ldexp(1.0, -24), n = 16 + p->D / 16 + 3;
  a.gamma = static_cast<float>(1.01 * n * u / (1.0 - n * u));
  a.ws = static_cast<char*>(workspace);
  a.L = L;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.col_cap = col_cap;
  a.dev_status = dev_status;
  *out = a;
  return SA_OK;
}

}  // namespace
}  // namespace sa

extern "C" {

sa_status sa_route(const sa_params* p, const void* q, const void* k, int32_t* row_ptr,
                   int32_t* col_idx, int64_t col_cap, void* workspace, size_t ws_bytes,
                   int32_t* dev_status, void* stream) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!q || !k || !row_ptr || !col_idx) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k)) return SA_ERR_INVALID_ARG;
  RouteArgs a;
  s = route_args(p, q, k, row_ptr, col_idx, col_cap, workspace, ws_bytes, dev_status, &a);
  if (s != SA_OK) return s;
  return from_cuda(launch_route(a, static_cast<cudaStream_t>(stream)));
}

sa_status sa_qk_prologue(const sa_params* p, const void* q_in, const void* k_in,
                         const float* gamma_q, const float* gamma_k, float eps,
                         const float* rope_cos, const float* rope_sin, void* q_out, void* k_out,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!q_in || !k_in || !q_out || !k_out) return SA_ERR_INVALID_ARG;
  if (!aligned16(q_in) || !aligned16(k_in) || !aligned16(q_out) || !aligned16(k_out))
    return SA_ERR_INVALID_ARG;
  if ((gamma_q && !aligned16(gamma_q)) || (gamma_k && !aligned16(gamma_k))) return SA_ERR_INVALID_ARG;
  if ((rope_cos == nullptr) != (rope_sin == nullptr)) return SA_ERR_INVALID_ARG;
  if (rope_cos && (!aligned16(rope_cos) || !aligned16(rope_sin))) return SA_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return SA_ERR_INVALID_ARG;
  RouteArgs a;
  s = route_args(p, q_in, k_in, nullptr, nullptr, 0, workspace, ws_bytes, dev_status, &a);
  if (s != SA_OK) return s;
  PrologueArgs pa{};
  pa.gamma_q = gamma_q;
  pa.gamma_k = gamma_k;
  pa.cos = rope_cos;
  pa.sin = rope_sin;
  pa.eps = eps;
  pa.q_out = static_cast<uint16_t*>(q_out);
  pa.k_out = static_cast<uint16_t*>(k_out);
  return from_cuda(launch_pool(a, &pa, static_cast<cudaStream_t>(stream)));
}

sa_status sa_route_pooled(const sa_params* p, int32_t* row_ptr, int32_t* col_idx,
                          int64_t col_cap, void* workspace, size_t ws_bytes, int32_t* dev_status,
                          void* stream) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!row_ptr || !col_idx) return SA_ERR_INVALID_ARG;
  RouteArgs a;
  s = route_args(p, nullptr, nullptr, row_ptr, col_idx, col_cap, workspace, ws_bytes, dev_status,
                 &a);
  if (s != SA_OK) return s;
  return from_cuda(launch_route_select(a, static_cast<cudaStream_t>(stream)));
}

sa_status sa_qk_quantize(const sa_params* p, const void* q, const void* k, uint8_t* q8,
                         uint8_t* k8, int8_t* q_exp, int8_t* k_exp, int32_t* dev_status,
                         void* stream) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (p->D != 128) return SA_ERR_UNSUPPORTED;
  if (!q || !k || !q8 || !k8 || !q_exp || !k_exp) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(q8) & 7u) != 0 ||
      (reinterpret_cast<uintptr_t>(k8) & 7u) != 0)
    return SA_ERR_INVALID_ARG;
  if (!strides_ok(p->q_stride) || !strides_ok(p->k_stride)) return SA_ERR_INVALID_ARG;
  QuantArgs qa{};
  qa.q = static_cast<const uint16_t*>(q);
  qa.k = static_cast<const uint16_t*>(k);
  for (int i = 0; i < 3; ++i) {
    qa.qs[i] = p->q_stride[i];
    qa.ks[i] = p->k_stride[i];
  }
  qa.q8 = q8;
  qa.k8 = k8;
  qa.y_stride[0] = static_cast<int64_t>(p->S) * p->H * p->D;
  qa.y_stride[1] = static_cast<int64_t>(p->H) * p->D;
  qa.y_stride[2] = p->D;
  qa.q_exp = q_exp;
  qa.k_exp = k_exp;
  qa.B = p->B;
  qa.S = p->S;
  qa.H = p->H;
  qa.Nb = num_blocks(p->S);
  qa.dev_status = dev_status;
  return from_cuda(launch_quant(qa, static_cast<cudaStream_t>(stream)));
}

sa_status sa_attn_sparse(const sa_params* p, const void* q, const void* k, const void* v,
                         const int32_t* row_ptr, const int32_t* col_idx, void* o, float* lse,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return attn_common(p, q, k, v, row_ptr, col_idx, o, lse, workspace, ws_bytes, dev_status, stream,
                     false);
}

sa_status sa_attn_prepare(const sa_params* p, const void* v, const int32_t* row_ptr,
                          const int32_t* col_idx, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream) {
  const sa_status s = attn_check(p, nullptr, nullptr, v, row_ptr, col_idx, nullptr, workspace,
                                 ws_bytes, false, true, false);
  if (s != SA_OK) return s;
  return attn_prepare_launch(p, v, row_ptr, col_idx, workspace, dev_status,
                             static_cast<cudaStream_t>(stream), false);
}

sa_status sa_attn_run(const sa_params* p, const void* q, const void* k, const int32_t* row_ptr,
                      const int32_t* col_idx, void* o, float* lse, void* workspace,
                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  const sa_status s = attn_check(p, q, k, nullptr, row_ptr, col_idx, o, workspace, ws_bytes,
                                 false, false, true);
  if (s != SA_OK) return s;
  return attn_run_launch(p, q, k, row_ptr, col_idx, o, lse, workspace, dev_status,
                         static_cast<cudaStream_t>(stream), false);
}

sa_status sa_attn_dense(const sa_params* p, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* workspace, size_t ws_bytes, int32_t* dev_status,
                        void* stream) {
  return attn_common(p, q, k, v, nullptr, nullptr, o, lse, workspace, ws_bytes, dev_status, stream,
                     true);
}

sa_status sa_forward_host(const sa_params* p, const void* q_host, const void* k_host,
                          const void* v_host, void* o_host, float* lse_host, void* q_dev,
                          void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int32_t* row_ptr,
                          int32_t* col_idx, int64_t col_cap, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream) {
  sa_status s = check_params(p);
  if (s != SA_OK) return s;
  if (!q_host || !k_host || !v_host || !o_host || !q_dev || !k_dev || !v_dev || !o_dev)
    return SA_ERR_INVALID_ARG;
  const int64_t cont[3] = {static_cast<int64_t>(p->S) * p->H * p->D,
                           static_cast<int64_t>(p->H) * p->D, p->D};
  for (int i = 0; i < 3; ++i)
    if (p->q_stride[i] != cont[i] || p->k_stride[i] != cont[i] || p->v_stride[i] != cont[i] ||
        p->o_stride[i] != cont[i])
      return SA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  HostPipe* hp = host_pipe(dev);
  if (!hp) return SA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hp->mu);

  // Head groups: group g's route and attention start as soon as its Q, K, V
  // slices are on the device and its O slice leaves as soon as it is done,
  // so the copies of one group overlap the compute of the others (H2D and
  // D2H on their own streams, compute on `stream`).
  // (lse is [B, H, S]: a head group's rows are one contiguous slice only for
  // B = 1, so a batched call that wants lse runs as a single group)
  // The groups shrink toward the end: a copy of a head slice moves rows of
  // (heads x D x 2) bytes, and the link carries wide rows faster (about 133
  // GB/s at 1 KB, 180 at 2 KB, 200 at 3.5 KB, 211 contiguous), so the first
  // groups are a quarter of the heads each; the last two (a seventh and the
  // rest) keep short the tail in which nothing is left to copy in.
  constexpr int kSched = 5;
  static_assert(kSched <= kHostGroups, "head-group schedule exceeds the events");
  const int G = ((p->B > 1 && lse_dev) || p->H < 16) ? 1 : kSched;
  const size_t row_bytes = static_cast<size_t>(p->H) * p->D * 2;   // one token, all heads
  const size_t rows = static_cast<size_t>(p->B) * p->S;
  // group boundaries at 0, 1/4, 1/2, 3/4, 25/28 and 1 of the heads
  auto head0 = [&](int g) {
    static const int num[kSched + 1] = {0, 7, 14, 21, 25, 28};
    return G == 1 ? (g == 0 ? 0 : p->H) : static_cast<int>((static_cast<int64_t>(p->H) * num[g] + 14) / 28);
  };
  if (cudaEventRecord(hp->start, st) != cudaSuccess ||
      cudaStreamWaitEvent(hp->h2d, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->d2h, hp->start, 0) != cudaSuccess)
    return SA_ERR_CUDA;
  for (int g = 0; g < G; ++g) {
    const size_t off = static_cast<size_t>(head0(g)) * p->D * 2;
    const size_t width = static_cast<size_t>(head0(g + 1) - head0(g)) * p->D * 2;
    const void* src[3] = {q_host, k_host, v_host};
    void* dst[3] = {q_dev, k_dev, v_dev};
    for (int t = 0; t < 3; ++t)
      if (cudaMemcpy2DAsync(static_cast<char*>(dst[t]) + off, row_bytes,
                            static_cast<const char*>(src[t]) + off, row_bytes, width, rows,
                            cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
        return SA_ERR_CUDA;
    if (cudaEventRecord(hp->in[g], hp->h2d) != cudaSuccess) return SA_ERR_CUDA;
  }
  for (int g = 0; g < G; ++g) {
    const int h0 = head0(g), h1 = head0(g + 1);
    sa_params pg = *p;
    pg.H = h1 - h0;
    const size_t off = static_cast<size_t>(h0) * p->D;                 // elements
    char* qg = static_cast<char*>(q_dev) + off * 2;
    char* kg = static_cast<char*>(k_dev) + off * 2;
    char* vg = static_cast<char*>(v_dev) + off * 2;
    char* og = static_cast<char*>(o_dev) + off * 2;
    float* lg = lse_dev ? lse_dev + static_cast<size_t>(h0) * p->S : nullptr;
    if (cudaStreamWaitEvent(st, hp->in[g], 0) != cudaSuccess) return SA_ERR_CUDA;
    s = sa_route(&pg, qg, kg, row_ptr, col_idx, col_cap, workspace, ws_bytes, dev_status, stream);
    if (s != SA_OK) return s;
    s = sa_attn_sparse(&pg, qg, kg, vg, row_ptr, col_idx, og, lg, workspace, ws_bytes,
                       dev_status, stream);
    if (s != SA_OK) return s;
    if (cudaEventRecord(hp->done[g], st) != cudaSuccess ||
        cudaStreamWaitEvent(hp->d2h, hp->done[g], 0) != cudaSuccess)
      return SA_ERR_CUDA;
    const size_t boff = static_cast<size_t>(h0) * p->D * 2;
    const size_t width = static_cast<size_t>(h1 - h0) * p->D * 2;
    if (cudaMemcpy2DAsync(static_cast<char*>(o_host) + boff, row_bytes,
                          static_cast<const char*>(o_dev) + boff, row_bytes, width, rows,
                          cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
      return SA_ERR_CUDA;
  }
  if (lse_host && lse_dev) {
    const size_t lb = static_cast<size_t>(p->B) * p->H * p->S * sizeof(float);
    if (cudaMemcpyAsync(lse_host, lse_dev, lb, cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
      return SA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->end, hp->d2h) != cudaSuccess ||
      cudaStreamWaitEvent(st, hp->end, 0) != cudaSuccess)
    return SA_ERR_CUDA;
  return SA_OK;
}

sa_status sa_dev_status_decode(int32_t d) {
  if (d & SA_DEV_TIMEOUT) return SA_ERR_TIMEOUT;
  if (d & SA_DEV_BAD_ROUTE) return SA_ERR_INVALID_ARG;
  if (d & SA_DEV_CAPACITY) return SA_ERR_CAPACITY;
  if (d & SA_DEV_RANGE) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

const char* sa_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_CAPACITY: return "SA_ERR_CAPACITY";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
    case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT";
  }
  return "SA_ERR_UNKNOWN";
}

}  // extern "C"
