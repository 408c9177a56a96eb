/*
 * sa.h -- C ABI of the GB300 (sm_103a) routed block-sparse self-attention
 * library (libsa_gb300.so).
 *
 * The layer: one packed sequence per batch entry, [B, S, H, D] bf16 Q/K/V
 * ("MiniMax H3 runs on single 4090 with 4.44x speedup over dense execution",
 * third paragraph: [1, 38247, 56, 128], tau = 1.0, diagonal, exact prefix
 * KV sink, compressed prefix queries; Sol-Engine H3-DataCenter release page,
 * policy paragraph: a 951-token exact prefix sink, no token reordering, the
 * first steps and layers dense).
 *
 * Conventions shared by every entry point:
 *  - Device pointers are device memory of the current CUDA device; host
 *    pointers are named *_host. The caller owns every buffer. The library
 *    never allocates device memory, frees or synchronises: every call
 *    enqueues work on `stream` (a cudaStream_t passed as void*; NULL = the
 *    legacy default stream) and returns (sa_forward_host also uses two copy
 *    streams of its own, see there).
 *  - The returned sa_status reports what can be checked before launch
 *    (arguments, support, launch errors). Conditions found on the device are
 *    OR-ed into *dev_status (an int32 in device memory that the caller sets
 *    to 0 before the first call and reads after the stream; NULL = do not
 *    report) as SA_DEV_* bits. The kernels never trap.
 *  - Tensors are [B, S, H, D] with the d index contiguous; the strides for
 *    b, s and h are given in elements and must be multiples of 8 (16 bytes),
 *    and every tensor base must be 16-byte aligned.
 *  - Query and key blocks are contiguous 64-token ranges; Nb = ceil(S/64);
 *    the last block holds S - 64 (Nb - 1) valid tokens. Tokens at or beyond S
 *    never contribute (the padding contributes exactly zero: "Making
 *    MiniMax-H3 up to 9x faster on H100s", section "The benchmark was not the
 *    product").
 */
#ifndef SA_GB300_H
#define SA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* a NULL pointer, a bad size, stride or alignment   */
  SA_ERR_UNSUPPORTED = 2, /* a valid request this build does not serve (D)     */
  SA_ERR_CAPACITY = 3,    /* a buffer or workspace is smaller than required    */
  SA_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed              */
  SA_ERR_TIMEOUT = 5      /* (decoded from dev_status) a bounded wait expired  */
} sa_status;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  SA_DEV_CAPACITY = 1 << 0, /* the route had more than col_cap entries; the
                               CSR is truncated (row_ptr is still exact)      */
  SA_DEV_TIMEOUT = 1 << 1,  /* a bounded pipeline wait gave up; the output of
                               the affected tiles is undefined                */
  SA_DEV_BAD_ROUTE = 1 << 2,/* sa_attn_sparse met a CSR that breaks its
                               contract (see sa_attn_sparse for what is then
                               attended)                                      */
  SA_DEV_RANGE = 1 << 3     /* a V value does not fit fp16 (|v| > 65504); the
                               P.V product runs in fp16, see sa_attn_sparse    */
};

/* Arithmetic of the attention's score product Q.K^T (sa_attn_*). */
enum {
  SA_QK_BF16 = 0,   /* bf16 x bf16 -> fp32 (the default)                       */
  SA_QK_FP8 = 1     /* 8-bit scores: Q and K quantised to e4m3 per (batch,
                       head, 64-token block) with power-of-two scales, see
                       sa_qk_quantize; D = 128 only                           */
};

/* Readings of the router rule (sa_route; the pages leave the rule open). */
enum {
  SA_ROUTE_THRESHOLD = 0,           /* keep p_ij >= tau / Nb (the default)     */
  SA_ROUTE_DENSE_PREFIX_QUERIES = 1,/* as THRESHOLD, and every query block that
                                       meets the prefix keeps every key block */
  SA_ROUTE_TOP_MASS = 2             /* keep the fewest key blocks of largest
                                       p_ij whose summed p_ij reaches tau     */
};

typedef struct sa_params {
  int32_t B, S, H, D;     /* D must be 64 or 128; B, S, H >= 1               */
  int32_t block;          /* must be 64                                       */
  int32_t prefix_len;     /* P, 0 <= P <= S: key tokens [0, P) are always
                             attended, via every key block j < ceil(P/64)    */
  float tau;              /* router parameter, >= 0: for THRESHOLD and
                             DENSE_PREFIX_QUERIES a multiple of the uniform
                             share (0 keeps every block); for TOP_MASS a mass
                             in [0, 1] (0 keeps only the forced blocks)      */
  float softmax_scale;    /* 0 => 1/sqrt(D); used for routing and attention  */
  int64_t q_stride[3];    /* element strides of b, s, h (d is contiguous)    */
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];
  int32_t route_mode;     /* SA_ROUTE_*; sa_params_init sets THRESHOLD       */
  int32_t q_block;        /* query block of the route: 0 or 64 (square, the
                             default) or 128 (two key blocks); see sa_route  */
  int32_t qk_format;      /* SA_QK_*; sa_params_init sets SA_QK_BF16         */
} sa_params;

/* Fills p for a contiguous [B, S, H, D] layout of all four tensors, with
 * route_mode = SA_ROUTE_THRESHOLD, q_block = 0, qk_format = SA_QK_BF16 and
 * softmax_scale = 0. */
void sa_params_init(sa_params* p, int32_t B, int32_t S, int32_t H, int32_t D,
                    int32_t prefix_len, float tau);

/* Nb = ceil(S / 64) (0 on bad params). */
int32_t sa_num_blocks(const sa_params* p);

/* Number of CSR rows, B*H*Nb; row_ptr holds this + 1 entries. */
int64_t sa_route_rows(const sa_params* p);

/* Worst-case number of route entries, B*H*Nb*Nb (every block kept). */
int64_t sa_route_max_nnz(const sa_params* p);

/* Bytes of device workspace sa_route needs (256-byte aligned start). */
size_t sa_route_workspace_bytes(const sa_params* p);

/*
 * sa_route -- the online router: for every (b, h, query block i) the
 * ascending list of key blocks that query block i attends.
 *
 * Rule (the pages name an online router with threshold tau over compressed
 * queries and keys, a diagonal threshold and an exact prefix sink; the exact
 * formula is this library's reading of them):
 *   qbar_i, kbar_j = mean of the valid Q / K tokens of block i / j;
 *   s_ij = softmax_scale * qbar_i . kbar_j for every key block j;
 *   p_ij = softmax over j of s_ij;
 *   keep j  iff  p_ij >= tau / Nb,  or j < ceil(P/64) (sink),  or j == i.
 * p->route_mode selects another reading: DENSE_PREFIX_QUERIES also keeps
 * every key block of query blocks i < ceil(P/64); TOP_MASS replaces the
 * first test by: rank the key blocks by p_ij descending (equal p_ij: lower j
 * first) and keep block j iff the blocks ranked above it sum to less than
 * tau.
 * p->q_block = 128 (any mode) routes 128-token query blocks over the same
 * 64-token key blocks: qbar_i is the mean of the valid tokens of query
 * tokens [128 i, 128 i + 128), the threshold is still tau / Nb with Nb the
 * number of key blocks, the diagonal of query block i is key blocks 2i and
 * 2i + 1, and DENSE_PREFIX_QUERIES covers query blocks i < ceil(P/128). The
 * CSR keeps one row per 64-token block: rows 2i and 2i + 1 both hold query
 * block i's list, so sa_attn_sparse reads it unchanged.
 * Decisions match an fp64 evaluation of the rule except on ties: for
 * THRESHOLD, |p_ij * Nb / tau - 1| <= 1e-6; for TOP_MASS, a preceding mass
 * within 1e-6 of tau, or p_ij within a relative 1e-6 of the last kept
 * block's across the cut. Pooling is exact to fp64 rounding; the scores are computed in fp32
 * and every row holding a decision inside a rigorous fp32 error bound is
 * recomputed in fp64.
 *
 * q, k       device, bf16 [B, S, H, D] with the strides in p; not modified.
 * row_ptr    device int32 [B*H*Nb + 1]; row r = (b*H + h)*Nb + i.
 *            row_ptr[0] = 0, row_ptr[r+1] - row_ptr[r] = entries of row r.
 * col_idx    device int32 [col_cap]; the key blocks of row r, ascending, at
 *            col_idx[row_ptr[r] .. row_ptr[r+1]).
 * col_cap    capacity of col_idx. If the route is longer, entries beyond
 *            col_cap are dropped and SA_DEV_CAPACITY is raised; passing
 *            sa_route_max_nnz(p) can never overflow.
 * workspace  device scratch of at least sa_route_workspace_bytes(p) bytes,
 *            256-byte aligned; its contents on entry do not matter.
 * Errors: SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED / SA_ERR_CAPACITY (ws
 * too small) before launch; SA_ERR_CUDA if a launch fails.
 */
sa_status sa_route(const sa_params* p, const void* q, const void* k,
                   int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                   void* workspace, size_t ws_bytes, int32_t* dev_status,
                   void* stream);

/* Size of the library-owned device scratch array sa_route_static runs on. */
#define SA_ROUTE_STATIC_WS_BYTES (32u << 20) /* 32 MiB */

/*
 * sa_route_static -- sa_route for callers that cannot allocate device
 * memory. The pages have no counterpart to this entry point; it exists for
 * callers such as a plugin inside an inference engine that has already
 * reserved all of HBM for its own pool, or code on a latency-critical path
 * where a cudaMalloc would synchronise the device.
 *
 * It computes exactly what sa_route computes (same kernels, same result) but
 * takes no workspace: the scratch lives in a fixed device array of
 * SA_ROUTE_STATIC_WS_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits. It allocates nothing and frees
 * nothing. The caller still passes q, k, row_ptr, col_idx (as for sa_route).
 *
 * Limits and behaviour:
 *  - Shapes whose sa_route_workspace_bytes(p) exceeds SA_ROUTE_STATIC_WS_BYTES
 *    are rejected with SA_ERR_CAPACITY before anything is launched. With
 *    D = 128 and 64-token query blocks the limit is 9 heads at S = 38,247,
 *    72 at S = 8,192 and 1 at S = 112,640 (15, 101 and 3 heads with
 *    q_block = 128); sa_route_workspace_bytes gives the need of any shape.
 *  - The first call on each device, made with that device current, looks up
 *    the array's device address and caches it; make that first call before
 *    any stream capture.
 *  - Every call on a device uses the same array and finds the previous call's
 *    contents there; what must start at zero is cleared by each call. Calls
 *    whose work overlaps on the GPU (e.g. on two unordered streams) race on
 *    the array and give undefined routes: order them on one stream.
 * Errors: as sa_route, plus SA_ERR_CAPACITY for shapes beyond the limit and
 * SA_ERR_CUDA if the array's address cannot be obtained.
 */
sa_status sa_route_static(const sa_params* p, const void* q, const void* k,
                          int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                          int32_t* dev_status, void* stream);

/*
 * sa_qk_prologue -- QK-norm + RoPE of q and k with the router's pooling
 * fused in (the fused QK-norm plus RoPE kernel of "Making MiniMax-H3 up to
 * 9x faster on H100s", section "Custom kernels"; the formulas are this
 * library's reading of that step). For every (b, token t, h) vector x [D]
 * of q_in (weights gamma_q) and of k_in (weights gamma_k):
 *   y_d = x_d / sqrt(mean_d(x_d^2) + eps) * gamma_d
 *   (y_2i, y_2i+1) -> (y_2i c - y_2i+1 s, y_2i s + y_2i+1 c),
 *       c = rope_cos[t][i], s = rope_sin[t][i]
 * computed in fp32 and rounded once to bf16 into q_out / k_out. The block
 * means of those bf16 outputs are written into `workspace` exactly as
 * sa_route would compute them from q_out, k_out; sa_route_pooled then
 * routes from them, so q_out and k_out are not read again for routing.
 *
 * q_in, k_in   device bf16 [B, S, H, D], strides p->q_stride / p->k_stride.
 * q_out, k_out device bf16, the same strides as q_in / k_in; each may be
 *              the same buffer as its input (in place) but must not
 *              otherwise overlap it.
 * gamma_q,     device fp32 [D], 16-byte aligned, or NULL for all ones.
 * gamma_k
 * eps          >= 0, added to the mean square.
 * rope_cos,    device fp32 [S][D/2] (row t = token t of the packed
 * rope_sin     sequence, any 1-D or 3-D rotary scheme), 16-byte aligned;
 *              both NULL for no rotation.
 * workspace    the route workspace, sa_route_workspace_bytes(p) bytes,
 *              256-byte aligned; p->q_block sets the query pooling.
 * Errors: as sa_route (SA_ERR_INVALID_ARG also for a bad eps, an unaligned
 * weight or table, or only one of the two tables).
 */
sa_status sa_qk_prologue(const sa_params* p, const void* q_in, const void* k_in,
                         const float* gamma_q, const float* gamma_k, float eps,
                         const float* rope_cos, const float* rope_sin, void* q_out,
                         void* k_out, void* workspace, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/*
 * sa_route_pooled -- sa_route from the block means that sa_qk_prologue left
 * in `workspace` (steps after pooling: logits, selection, fp64 recheck,
 * CSR). p must give the same B, S, H, D, q_block and strides as that
 * sa_qk_prologue call (prefix_len, tau, route_mode and softmax_scale may
 * differ); the workspace's contents are not checked. The result equals
 * sa_route on the prologue's q_out, k_out. Arguments and errors as sa_route.
 */
sa_status sa_route_pooled(const sa_params* p, int32_t* row_ptr, int32_t* col_idx,
                          int64_t col_cap, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream);

/*
 * sa_qk_quantize -- the 8-bit copies of q and k that sa_attn_* use with
 * p->qk_format = SA_QK_FP8 (MiniAcc blog, "What is SageAttention?": the
 * score computation in 8-bit arithmetic; the format and scaling are this
 * library's reading: FP8 e4m3, the 8-bit format GB300's tensor cores run
 * fastest). For every (b, h, 64-token block j) of q, and of k:
 *   e     = the smallest integer with amax / 2^e <= 448, where amax is the
 *           largest |x| over the block's valid tokens and all D (e = 0 for
 *           an all-zero block);
 *   code  = x / 2^e rounded to the nearest e4m3 value, ties to even
 *           (exact scaling: the scale is a power of two).
 * The attention's logits are then scale * 2^(e_q + e_k) * (codes_q . codes_k).
 *
 * q, k          device bf16 [B, S, H, D] (strides in p), D = 128.
 * q8, k8        device uint8 [B, S, H, D], contiguous, 8-byte aligned: the
 *               e4m3 codes (tokens >= S are not written).
 * q_exp, k_exp  device int8 [B*H*Nb]: e of block (b, h, j) at (b*H + h)*Nb + j.
 * A non-finite input raises SA_DEV_RANGE (its block's codes are undefined).
 * Errors: SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED (D != 128) before launch.
 */
sa_status sa_qk_quantize(const sa_params* p, const void* q, const void* k, uint8_t* q8,
                         uint8_t* k8, int8_t* q_exp, int8_t* k_exp, int32_t* dev_status,
                         void* stream);

/* Bytes of device workspace sa_attn_sparse / sa_attn_dense need (more with
 * p->qk_format = SA_QK_FP8: the codes of Q and K live there). */
size_t sa_attn_workspace_bytes(const sa_params* p);

/*
 * sa_attn_sparse -- block-sparse attention forward over a route: only the
 * routed (query block, key block) pairs are computed (MiniAcc blog, "What is
 * Sol attention?"), each exactly (exact softmax over the selected keys).
 *
 * For every query token t of block i (head h, batch b), over the valid key
 * tokens u of the key blocks listed for row (b, h, i):
 *   l_u = softmax_scale * q_t . k_u,   a_u = exp(l_u - max l) / sum exp(.),
 *   o_t = sum_u a_u v_u,              lse_t = max l + log sum exp(l - max l).
 * Only the listed K/V blocks are read. A row with an empty list gives o = 0
 * and lse = -inf.
 *
 * Precision: Q.K^T is a bf16 x bf16 product with fp32 accumulation (with
 * p->qk_format = SA_QK_FP8: an e4m3 x e4m3 product of sa_qk_quantize's codes,
 * fp32 accumulation, times the blocks' power-of-two scales; the codes are
 * made in the workspace by each call); the softmax is fp32; the P.V product
 * takes P and V in fp16 (V is repacked once per call into the workspace)
 * with fp32 accumulation; o is rounded once to bf16. |v| must be <= 65504
 * (else SA_DEV_RANGE).
 *
 * q, k, v    device bf16 [B, S, H, D] (strides in p); not modified.
 * row_ptr,   device int32 CSR as written by sa_route: row_ptr[B*H*Nb] = nnz
 * col_idx    entries in col_idx (which must hold at least that many), each
 *            row strictly ascending with entries in [0, Nb). A CSR that
 *            breaks this raises SA_DEV_BAD_ROUTE and is attended as follows:
 *            a row whose span [row_ptr[r], row_ptr[r+1]) does not lie inside
 *            [0, nnz] or is longer than Nb is skipped whole (its query rows
 *            give o = 0, lse = -inf; col_idx is not read for it); entries
 *            outside [0, Nb) are skipped; a row that is not strictly
 *            ascending (a repeated entry included) is attended as the set of
 *            its entries. Nothing is read outside col_idx[0, nnz).
 * o          device bf16 [B, S, H, D] (o_stride); rows >= S are not written.
 * lse        device fp32 [B, H, S] (natural log), or NULL.
 * workspace  device scratch of sa_attn_workspace_bytes(p) bytes, 256-byte
 *            aligned.
 * Each 128-row tile of the kernel holds two 64-token query blocks of one
 * head. With p->q_block = 0 or 64 the pairs are chosen per call from the
 * route (largest key-list overlap, among blocks at most 32 apart); with
 * p->q_block = 128 the tiles are the 128-token query blocks (2i, 2i + 1),
 * which share their key list when the route came from sa_route with the
 * same q_block (any CSR is still attended exactly).
 */
sa_status sa_attn_sparse(const sa_params* p, const void* q, const void* k,
                         const void* v, const int32_t* row_ptr,
                         const int32_t* col_idx, void* o, float* lse,
                         void* workspace, size_t ws_bytes, int32_t* dev_status,
                         void* stream);

/*
 * sa_attn_prepare, sa_attn_run -- sa_attn_sparse in two calls, with the same
 * result: sa_attn_prepare repacks V into the workspace and (for 64-token
 * query blocks) chooses the tile pairs from the route; sa_attn_run launches
 * the attention kernel over that workspace (with SA_QK_FP8, after quantising
 * q and k into it, as sa_qk_quantize does). Between them the caller may
 * enqueue other work (or time the kernel alone); sa_attn_run must see the
 * same p, route and workspace, after sa_attn_prepare on the same stream (or
 * ordered after it), and V unchanged. Arguments and errors as
 * sa_attn_sparse, each call checking what it takes.
 */
sa_status sa_attn_prepare(const sa_params* p, const void* v, const int32_t* row_ptr,
                          const int32_t* col_idx, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream);
sa_status sa_attn_run(const sa_params* p, const void* q, const void* k,
                      const int32_t* row_ptr, const int32_t* col_idx, void* o, float* lse,
                      void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * sa_attn_dense -- the same forward with every key block attended (density
 * 100%), as the pages run for the first denoising steps and the first layers
 * (Sol-Engine H3-DataCenter release page, policy paragraph). Arguments as in
 * sa_attn_sparse, without the route.
 */
sa_status sa_attn_dense(const sa_params* p, const void* q, const void* k,
                        const void* v, void* o, float* lse, void* workspace,
                        size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * sa_forward_host -- one whole layer from host memory: copies q, k, v
 * (host, pinned for asynchronous copies) to the device buffers, routes,
 * attends, and copies o (and lse if both lse pointers are non-NULL) back,
 * then returns without synchronising. The work is split into groups of
 * heads (for H >= 16 five groups, a quarter of the heads each and then a
 * seventh and the rest, since wide head slices copy faster and narrow last
 * groups shorten the tail; one group for H < 16 or for B > 1 with lse):
 * each group is routed and attended as soon as its q, k, v slices have
 * landed, and its o slice is copied back as soon as it is done, so the
 * copies overlap the compute. Compute runs on `stream`; the copies run on two
 * streams the library creates, with a few events, on the first call on each
 * device and keeps until the process exits. All of it is ordered after the
 * work enqueued on `stream` before the call and before the work enqueued on
 * it after the call. Calls on one device from several host threads are
 * serialised by the library. Every device buffer is the caller's, sized as
 * for sa_route / sa_attn_sparse, with q_dev, k_dev, v_dev, o_dev laid out
 * with the strides in p and *_host contiguous copies of the same
 * [B, S, H, D] extents (the strides in p must then describe a contiguous
 * tensor). The route workspace and the attention workspace may be the same
 * buffer if it is large enough for both.
 */
sa_status sa_forward_host(const sa_params* p, const void* q_host,
                          const void* k_host, const void* v_host, void* o_host,
                          float* lse_host, void* q_dev, void* k_dev,
                          void* v_dev, void* o_dev, float* lse_dev,
                          int32_t* row_ptr, int32_t* col_idx, int64_t col_cap,
                          void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream);

/*
 * sa_check_wait_timeout -- a device check of the failure path that every
 * pipeline wait of this library shares (no counterpart on the pages): it
 * launches one warp that waits on a barrier nothing completes. The wait gives
 * up after the library's time limit (250 ms), OR-s SA_DEV_TIMEOUT into
 * *dev_status (device memory, required) and the kernel returns; the context
 * stays usable. Nothing faults, traps or hangs. Asynchronous on `stream`.
 */
sa_status sa_check_wait_timeout(int32_t* dev_status, void* stream);

/* Decodes *dev_status bits into the most severe sa_status (SA_OK if 0). */
sa_status sa_dev_status_decode(int32_t dev_status);

/* A static, NUL-terminated name of the status. */
const char* sa_status_string(sa_status s);

#ifdef __cplusplus
}
#endif

#endif /* SA_GB300_H */
