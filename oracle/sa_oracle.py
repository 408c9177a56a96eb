"""CPU oracle for routed block-sparse self-attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module. The CUDA library never calls it, and it shares no
code with the CUDA library: it is a plain, slow, fp64 restatement of what the
layer computes, written so that a reader can check it against the pages by eye.

What the pages fix, and where:

* "MiniMax H3 runs on single 4090 with 4.44x speedup over dense execution",
  third paragraph: the layer attends over a [1, 38247, 56, 128] bf16 tensor;
  Sol-Attn runs with tau = 1.0, a diagonal threshold, an exact KV sink for the
  prefix and compressed prefix queries; the first steps and layers run dense.
  (The Hebrew version of the same article, same paragraph, reads the garbled
  "KV queue" as an exact KV *sink* and "full compression" as full *density*.)
* Sol-Engine H3-DataCenter release page, policy paragraph: the first 10 steps
  and first two layers stay dense; tau = 1.0; no token reordering; an exact
  951-token multimodal prefix sink; the same online routing on every backend.
* "Making MiniMax-H3 up to 9x faster on H100s", section "The benchmark was not
  the product": the sequence is padded to a 64-token multiple and the padding
  must contribute exactly zero.
* MiniAcc blog, section "What is Sol attention?": Sol picks promising pairs per
  head and computes only those.

The pages give no router formula. The reading used here (step numbers follow
the docstrings below):

1. bf16 -> fp64 (exact).
2. Blocks are contiguous 64-token ranges; Nb = ceil(S/64); block j has
   n_j = min(64, S - 64 j) valid tokens.
3. Pool ("compressed" queries/keys): the arithmetic mean of the valid tokens.
4. Pooled logits s_ij = scale * qbar_i . kbar_j over all Nb key blocks,
   scale = 1/sqrt(D) unless given.
5. p_ij = softmax_j(s_ij).
6. Keep j iff p_ij >= tau / Nb (at or above tau times the uniform share), OR
   j is a sink block (64 j < P), OR j == i (the diagonal).
7. Attention of every query token of block i over the valid tokens of the
   kept key blocks: exact softmax(scale * q.k) weighted sum of V, and the
   log-sum-exp of the scaled logits. Non-causal. Padding tokens never enter.
8. Dense attention = step 7 with every block kept.

Other readings of the router (the pages leave the rule open; none is the
default):

* ``mode="dense_prefix_queries"``: step 6 as above, and every query block
  that intersects the prefix attends every key block (a reading of
  "compressed prefix queries" in which the prefix rows are not routed at all).
* ``mode="top_mass"``: step 6 keeps, besides the sink and the diagonal, the
  smallest set of key blocks of largest p whose summed p reaches tau (tau a
  mass in [0, 1]): blocks are ranked by p descending, equal p by index
  ascending, and the block of rank r is kept iff the blocks ranked above it
  hold less than tau (MiniAcc blog, "What is Sol attention?": Sol keeps the
  promising pairs of each head). Cumulative sums within 1e-6 of tau, and p
  within a relative 1e-6 of the last kept block's across the cut, are ties.
* ``q_block=128`` (non-square blocks, with any mode): query blocks of 128
  tokens over key blocks of 64. Step 3 pools each query block over its own
  valid tokens (up to 128), step 4 scores it against every 64-token key
  block, step 6 compares with tau / Nb (Nb the number of key blocks) and
  forces, besides the sink columns, the key blocks inside the query block
  (its diagonal: key blocks 2i and 2i + 1). A query block meets the prefix
  when 128 i < P. The route is still stated per 64-token query block: both
  halves of a 128-token query block carry its key list, so step 7 is
  unchanged.

The step before attention, fused with the pooling ("Making MiniMax-H3 up to
9x faster on H100s", section "Custom kernels": a fused QK-norm plus RoPE
kernel). The page names the two operations only; the reading used here:

9. QK-norm: RMS normalisation of each (token, head) vector over its D dims,
   x_hat = x / sqrt(mean_d x_d^2 + eps) * gamma_d, with one weight vector
   gamma [D] for Q and one for K.
10. RoPE: each interleaved pair (2i, 2i + 1) of x_hat is rotated by the angle
    of token t and pair i, given as tables cos[t, i], sin[t, i]:
    (a, b) -> (a cos - b sin, a sin + b cos). 1-D and 3-D (video) rotary
    schemes differ only in the tables.
11. The router then pools the rounded (bf16) outputs, as in step 3.

8-bit score computation (MiniAcc blog, "What is SageAttention?": the
attention's score computation runs in 8-bit arithmetic instead of 16-bit;
the page names no format or scaling; the reading used here, for FP8 e4m3,
the 8-bit format GB300's tensor cores run fastest):

12. Q and K are quantised per (batch, head, 64-token block): the block's
    scale is 2^e with e the smallest integer such that amax / 2^e <= 448
    (amax = the largest |x| over the block's valid tokens and all D; e = 0
    for an all-zero block), and every x / 2^e is rounded to the nearest e4m3
    value, ties to even (bias 7, three mantissa bits, subnormals below 2^-6,
    largest finite value 448). Power-of-two scales keep x / 2^e exact, so the
    rounding is the only approximation.
13. Attention is step 7 with the logits of the dequantised Q and K
    (code * 2^e); V, the softmax and the route are unchanged.

The parity of a Sol "correction term" for skipped pairs (MiniAcc blog, same
section) is not pinned: the pages give no formula and it is not applied.
"""

from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 64
Q_BLOCKS = (64, 128)      # query block sizes of the router readings
TIE_WINDOW = 1e-6


def as_f64(x) -> np.ndarray:
    """Step 1: exact conversion of a bf16 torch tensor (or any array) to fp64."""
    if hasattr(x, "detach"):  # torch tensor; bf16 -> fp32 -> fp64 is exact
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def num_blocks(S: int, block: int = BLOCK) -> int:
    return (S + block - 1) // block


def block_bounds(S: int, block: int = BLOCK) -> Tuple[np.ndarray, np.ndarray]:
    """Step 2: start token and valid-token count of each block."""
    nb = num_blocks(S, block)
    starts = np.arange(nb, dtype=np.int64) * block
    counts = np.minimum(block, S - starts)
    return starts, counts


def pool_blocks(x: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """Step 3: mean over the valid tokens of each block.

    x: [B, S, H, D] fp64. Returns [B, H, Nb, D]. The partial last block is
    divided by its own token count, not by 64.
    """
    B, S, H, D = x.shape
    starts, counts = block_bounds(S, block)
    out = np.empty((B, H, len(starts), D), dtype=np.float64)
    for j, (s0, n) in enumerate(zip(starts, counts)):
        out[:, :, j, :] = x[:, s0:s0 + n].sum(axis=1) / float(n)
    return out


def pooled_logits(qbar: np.ndarray, kbar: np.ndarray, scale: float) -> np.ndarray:
    """Step 4: s[b,h,i,j] = scale * qbar[b,h,i] . kbar[b,h,j] (all j)."""
    return scale * np.matmul(qbar, np.swapaxes(kbar, -1, -2))


def pooled_softmax(s: np.ndarray) -> np.ndarray:
    """Step 5: softmax over the key-block axis, max subtracted first."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def forced_mask(Nb: int, prefix_len: int, block: int = BLOCK,
                q_block: Optional[int] = None) -> np.ndarray:
    """Step 6, forced part: [Nq, Nb] bool, sink columns and the diagonal.

    Sink blocks are the key blocks that intersect the prefix [0, P), i.e.
    j < ceil(P/64); every prefix key is then attended with its exact weight.
    The diagonal of query block i is every key block inside it: j = i for
    square blocks, j in {2i, 2i + 1} (those that exist) for 128-token query
    blocks. Nq = ceil(Nb / (q_block / block)) (= Nb for square blocks).
    """
    q_block = block if q_block is None else q_block
    r = q_block // block
    Nq = (Nb + r - 1) // r
    n_sink = (prefix_len + block - 1) // block
    f = np.zeros((Nq, Nb), dtype=bool)
    f[:, :n_sink] = True
    for i in range(Nq):
        f[i, i * r:min(Nb, i * r + r)] = True
    return f


def select_blocks(p: np.ndarray, tau: float, prefix_len: int,
                  block: int = BLOCK, q_block: Optional[int] = None) -> np.ndarray:
    """Step 6: kept[b,h,i,j] = p >= tau/Nb, OR sink, OR diagonal."""
    Nb = p.shape[-1]
    kept = p >= (tau / Nb)
    return kept | forced_mask(Nb, prefix_len, block, q_block)


def select_top_mass(p: np.ndarray, tau: float) -> Tuple[np.ndarray, np.ndarray]:
    """Top-mass reading of step 6, without the forced blocks.

    For every row: rank the key blocks by p descending (equal p: lower index
    first); the block of rank r is kept iff the blocks ranked above it sum to
    less than tau. Returns (kept, ties), both [..., Nb] bool; ties marks the
    decisions another correct implementation may take either way: a block
    whose preceding mass is within 1e-6 of tau, and, when the p on either
    side of the cut differ by at most 1e-6 of the last kept block's p, the
    blocks whose p lies that close to the cut.
    """
    flat = p.reshape(-1, p.shape[-1])
    kept = np.zeros(flat.shape, dtype=bool)
    ties = np.zeros(flat.shape, dtype=bool)
    idx = np.arange(flat.shape[1])
    for r in range(flat.shape[0]):
        row = flat[r]
        order = np.lexsort((idx, -row))          # p descending, then index ascending
        before = np.concatenate([[0.0], np.cumsum(row[order])[:-1]])
        keep_rank = before < tau
        kept[r, order[keep_rank]] = True
        ties[r, order[np.abs(before - tau) <= TIE_WINDOW]] = True
        n_keep = int(keep_rank.sum())
        if 0 < n_keep < len(row):
            p_last, p_next = row[order[n_keep - 1]], row[order[n_keep]]
            w = TIE_WINDOW * p_last
            if p_last - p_next <= w:              # the order across the cut is ambiguous
                ties[r] |= (row >= p_next - w) & (row <= p_last + w)
    return kept.reshape(p.shape), ties.reshape(p.shape)


def threshold_ratio(p: np.ndarray, tau: float) -> np.ndarray:
    """p * Nb / tau: a block is kept by the router iff this is >= 1.

    Decisions with |ratio - 1| <= 1e-6 are ties that another correct
    implementation may take either way.
    """
    Nb = p.shape[-1]
    if tau == 0.0:
        return np.full_like(p, np.inf)
    return p * (Nb / tau)


def to_csr(kept: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Rows (b, h, i) in row-major order; columns ascending."""
    B, H, Nb, _ = kept.shape
    flat = kept.reshape(B * H * Nb, Nb)
    counts = flat.sum(axis=1)
    row_ptr = np.zeros(B * H * Nb + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    col_idx = np.nonzero(flat)[1].astype(np.int64)  # row-major scan: ascending per row
    return row_ptr, col_idx


ROUTE_MODES = ("threshold", "dense_prefix_queries", "top_mass")


def route_ref(q, k, prefix_len: int, tau: float, scale: Optional[float] = None,
              block: int = BLOCK, mode: str = "threshold",
              q_block: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Steps 1-6: the block route of every (b, h, query block).

    Returns kept [B,H,Nb,Nb] bool, the CSR (row_ptr, col_idx), the pooled
    softmax p, the forced mask (broadcast to kept's shape) and ties, the
    decisions another correct router may take either way (never forced
    ones). ``mode`` picks the reading of step 6 (module docstring).

    ``q_block`` (64 or 128, default the key block) is the query block size.
    Rows stay per 64-token block: with 128-token query blocks, rows 2i and
    2i + 1 are both the route of query block i (so are p, ratio, forced and
    ties); "kept_q" and "p_q" hold the [B,H,Nq,Nb] values per query block.
    """
    if mode not in ROUTE_MODES:
        raise ValueError(f"unknown route mode {mode!r}")
    q_block = block if q_block is None else int(q_block)
    if q_block not in Q_BLOCKS or q_block % block:
        raise ValueError(f"unsupported query block {q_block}")
    r = q_block // block
    qf, kf = as_f64(q), as_f64(k)
    D = qf.shape[-1]
    scale = 1.0 / math.sqrt(D) if not scale else scale
    qbar, kbar = pool_blocks(qf, q_block), pool_blocks(kf, block)
    del qf, kf
    p = pooled_softmax(pooled_logits(qbar, kbar, scale))      # [B, H, Nq, Nb]
    Nb = p.shape[-1]
    forced = np.broadcast_to(forced_mask(Nb, prefix_len, block, q_block), p.shape).copy()
    if mode == "dense_prefix_queries":
        n_prefix_q = (prefix_len + q_block - 1) // q_block    # query blocks meeting [0, P)
        forced[..., :n_prefix_q, :] = True
    if mode == "top_mass":
        by_mass, ties = select_top_mass(p, tau)
        kept = by_mass | forced
        ratio = None
    else:
        kept = select_blocks(p, tau, prefix_len, block, q_block) | forced
        ratio = threshold_ratio(p, tau)
        ties = np.abs(ratio - 1.0) <= TIE_WINDOW
    ties = ties & ~forced
    kept_q, p_q = kept, p
    if r > 1:                        # one row per 64-token block: repeat each query block's row
        rows = np.arange(Nb) // r
        kept, p, forced, ties = (x[..., rows, :] for x in (kept, p, forced, ties))
        ratio = None if ratio is None else ratio[..., rows, :]
    row_ptr, col_idx = to_csr(kept)
    return {"kept": kept, "row_ptr": row_ptr, "col_idx": col_idx, "p": p,
            "ratio": ratio, "forced": forced, "ties": ties, "qbar": qbar, "kbar": kbar,
            "kept_q": kept_q, "p_q": p_q, "q_block": q_block}


def block_density(kept: np.ndarray) -> float:
    return float(kept.mean())


def attend_rows(qf: np.ndarray, kf: np.ndarray, vf: np.ndarray, b: int, h: int,
                i: int, blocks: Sequence[int], scale: float,
                block: int = BLOCK) -> Tuple[np.ndarray, np.ndarray]:
    """Step 7 for query block i of head h: (O [n_i, D], LSE [n_i]) in fp64.

    The key set is the valid tokens of the listed key blocks, in sequence
    order; padding tokens (>= S) are never included, so they weigh exactly 0.
    """
    S = qf.shape[1]
    q0, q1 = i * block, min(S, i * block + block)
    if len(blocks) == 0:
        # An empty key set: the sum of exponentials is 0, so LSE = log 0 = -inf,
        # and the output is taken as 0 (an empty weighted sum).
        return np.zeros((q1 - q0, qf.shape[3])), np.full(q1 - q0, -np.inf)
    keys = np.concatenate([np.arange(j * block, min(S, j * block + block))
                           for j in sorted(blocks)])
    Q = qf[b, q0:q1, h, :]
    K = kf[b, keys, h, :]
    V = vf[b, keys, h, :]
    logits = scale * (Q @ K.T)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    z = e.sum(axis=1, keepdims=True)
    out = (e / z) @ V
    lse = (m + np.log(z))[:, 0]
    return out, lse


def _head_f64(x, b: int, h: int) -> np.ndarray:
    """Step 1 for one (batch, head) slice: [S, D] fp64."""
    if hasattr(x, "detach"):
        return x[b, :, h, :].detach().cpu().float().numpy().astype(np.float64)
    return np.asarray(x[b, :, h, :], dtype=np.float64)


def attn_ref(q, k, v, row_ptr: np.ndarray, col_idx: np.ndarray,
             scale: Optional[float] = None,
             items: Optional[Iterable[Tuple[int, int, int]]] = None,
             block: int = BLOCK):
    """Step 7 over a CSR route.

    Without ``items`` it returns the full O [B,S,H,D] and LSE [B,H,S] (fp64).
    With ``items`` (a list of (b, h, i)) it returns {(b, h, i): (O, LSE)} for
    just those query blocks.
    """
    B, S, H, D = q.shape
    Nb = num_blocks(S, block)
    scale = 1.0 / math.sqrt(D) if not scale else scale

    def blocks_of(b, h, i):
        r = (b * H + h) * Nb + i
        return [int(c) for c in col_idx[row_ptr[r]:row_ptr[r + 1]]]

    cache = {}

    def head(b, h):
        if (b, h) not in cache:
            cache.clear()
            cache[(b, h)] = tuple(_head_f64(x, b, h)[None, :, None, :] for x in (q, k, v))
        return cache[(b, h)]

    if items is not None:
        out = {}
        for (b, h, i) in sorted(items, key=lambda t: (t[0], t[1], t[2])):
            qf, kf, vf = head(b, h)
            out[(b, h, i)] = attend_rows(qf, kf, vf, 0, 0, i, blocks_of(b, h, i), scale, block)
        return out
    o = np.zeros((B, S, H, D), dtype=np.float64)
    lse = np.zeros((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            qf, kf, vf = head(b, h)
            for i in range(Nb):
                oi, li = attend_rows(qf, kf, vf, 0, 0, i, blocks_of(b, h, i), scale, block)
                q0 = i * block
                o[b, q0:q0 + oi.shape[0], h, :] = oi
                lse[b, h, q0:q0 + oi.shape[0]] = li
    return o, lse


def dense_csr(B: int, H: int, S: int, block: int = BLOCK) -> Tuple[np.ndarray, np.ndarray]:
    """Step 8: the route that keeps every key block of every row."""
    Nb = num_blocks(S, block)
    return to_csr(np.ones((B, H, Nb, Nb), dtype=bool))


def attn_dense_ref(q, k, v, scale: Optional[float] = None,
                   items: Optional[Iterable[Tuple[int, int, int]]] = None,
                   block: int = BLOCK):
    """Step 8: dense attention, i.e. step 7 with every block kept."""
    B, S, H, _ = q.shape
    row_ptr, col_idx = dense_csr(B, H, S, block)
    return attn_ref(q, k, v, row_ptr, col_idx, scale=scale, items=items, block=block)


def routed_flops(row_ptr: np.ndarray, col_idx: np.ndarray, B: int, H: int, S: int,
                 D: int, block: int = BLOCK) -> int:
    """Algorithmic work of step 7: 4*D*sum over routed (query block, key block)
    pairs of n_i * n_j (valid tokens only)."""
    Nb = num_blocks(S, block)
    _, counts = block_bounds(S, block)
    rows = np.arange(B * H * Nb)
    ni = counts[rows % Nb]
    cs = np.concatenate([[0], np.cumsum(counts[col_idx])])
    per_row = cs[row_ptr[1:]] - cs[row_ptr[:-1]]
    return int(4 * D * int((ni * per_row).sum()))


def tie_mask(ratio: np.ndarray, forced: np.ndarray) -> np.ndarray:
    """Decisions another correct router may take either way: router ties
    (|p Nb / tau - 1| <= 1e-6) on blocks that are not forced."""
    return (np.abs(ratio - 1.0) <= TIE_WINDOW) & ~forced


def qk_prologue_ref(x, gamma: Optional[np.ndarray], eps: float,
                    cos: Optional[np.ndarray], sin: Optional[np.ndarray]) -> np.ndarray:
    """Steps 9-10: QK-norm then RoPE of x [B, S, H, D] in fp64.

    gamma [D] (None: ones), cos/sin [S, D/2] (None: no rotation). Returns the
    exact result in fp64; the CUDA kernel rounds it once to bf16.
    """
    xf = as_f64(x)
    D = xf.shape[-1]
    ms = (xf * xf).mean(axis=-1, keepdims=True)
    y = xf / np.sqrt(ms + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    if cos is None:
        return y
    c = np.asarray(cos, dtype=np.float64)[None, :, None, :]      # [1, S, 1, D/2]
    s_ = np.asarray(sin, dtype=np.float64)[None, :, None, :]
    a, b = y[..., 0::2], y[..., 1::2]
    out = np.empty_like(y)
    out[..., 0::2] = a * c - b * s_
    out[..., 1::2] = a * s_ + b * c
    return out


# ------------------------------------------------------------------ FP8 --

E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """The value of an e4m3 byte (step 12's format): sign bit, four exponent
    bits with bias 7, three mantissa bits; exponent field 0 is subnormal
    (m/8 * 2^-6); the all-ones pattern S.1111.111 is NaN (no infinities)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    ef, m = (code >> 3) & 0xF, code & 0x7
    if ef == 0xF and m == 0x7:
        return float("nan")
    if ef == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (ef - 7)


def e4m3_round(x) -> np.ndarray:
    """Step 12: round fp64 values with |x| <= 448 to the nearest e4m3 value,
    ties to even. The spacing of e4m3 values in the binade [2^E, 2^(E+1)) is
    2^(E-3), and 2^-9 below 2^-6 (the subnormals share the first normal
    binade's spacing)."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, k = np.frexp(np.where(ax > 0, ax, 1.0))       # ax = f 2^k, f in [0.5, 1)
    E = np.maximum(k - 1, -6)                        # binade exponent, subnormals at -6
    ulp = np.ldexp(1.0, (E - 3).astype(np.int64))
    return np.round(x / ulp) * ulp                   # numpy rounds half to even


def e4m3_encode(v) -> np.ndarray:
    """The e4m3 byte of values already on the e4m3 grid (inverse of
    e4m3_decode for finite values; -0 is encoded as +0)."""
    v = np.asarray(v, dtype=np.float64)
    av = np.abs(v)
    _, k = np.frexp(np.where(av > 0, av, 1.0))
    E = k - 1
    sub = av < 2.0 ** -6
    ef = np.where(sub, 0, E + 7)
    m = np.where(sub, av / 2.0 ** -9, (av / np.ldexp(1.0, E.astype(np.int64)) - 1.0) * 8.0)
    code = (ef.astype(np.int64) << 3) | np.rint(m).astype(np.int64)
    code = np.where(av == 0, 0, code)
    return (code | np.where(v < 0, 0x80, 0)).astype(np.uint8)


def fp8_block_exponent(amax: float) -> int:
    """Step 12: the smallest integer e with amax / 2^e <= 448 (0 for amax = 0).
    With amax = f 2^k, f in [0.5, 1) and 448 = 0.875 * 2^9: e = k - 9, plus
    one when f > 0.875."""
    if amax == 0:
        return 0
    f, k = math.frexp(float(amax))
    return int(k - 9 + (1 if f > 0.875 else 0))


def quantize_qk_ref(x, heads: Optional[Sequence[int]] = None, block: int = BLOCK):
    """Step 12 for a [B, S, H, D] tensor: returns (codes uint8 [B, S, Hs, D],
    exponents int [B, Hs, Nb], dequantised values fp64 [B, S, Hs, D]) for the
    heads in ``heads`` (all heads if None, in that order)."""
    B, S, H, D = x.shape
    heads = list(range(H)) if heads is None else list(heads)
    Nb = num_blocks(S, block)
    codes = np.zeros((B, S, len(heads), D), dtype=np.uint8)
    exps = np.zeros((B, len(heads), Nb), dtype=np.int64)
    deq = np.zeros((B, S, len(heads), D), dtype=np.float64)
    for b in range(B):
        for hi, h in enumerate(heads):
            xf = _head_f64(x, b, h)
            for j in range(Nb):
                t0, t1 = j * block, min(S, j * block + block)
                blk = xf[t0:t1]
                e = fp8_block_exponent(np.abs(blk).max())
                grid = e4m3_round(blk / 2.0 ** e)
                exps[b, hi, j] = e
                codes[b, t0:t1, hi, :] = e4m3_encode(grid)
                deq[b, t0:t1, hi, :] = grid * 2.0 ** e
    return codes, exps, deq


def attn_fp8_ref(q, k, v, row_ptr: np.ndarray, col_idx: np.ndarray,
                 scale: Optional[float] = None,
                 items: Optional[Iterable[Tuple[int, int, int]]] = None,
                 block: int = BLOCK):
    """Step 13: step 7 over a CSR route with the logits of the dequantised Q
    and K of step 12 (V unchanged). With ``items`` only their heads are
    quantised; returns what attn_ref returns."""
    B, S, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if not scale else scale
    heads = sorted({h for (_, h, _) in items}) if items is not None else list(range(H))
    _, _, qd = quantize_qk_ref(q, heads, block)
    _, _, kd = quantize_qk_ref(k, heads, block)
    qf = np.zeros((B, S, H, D)) if items is None else None
    if items is None:
        kf = np.zeros((B, S, H, D))
        qf[:, :, heads, :] = qd
        kf[:, :, heads, :] = kd
        return attn_ref(qf, kf, v, row_ptr, col_idx, scale=scale, block=block)
    Nb = num_blocks(S, block)
    out = {}
    for (b, h, i) in items:
        hi = heads.index(h)
        vf = _head_f64(v, b, h)[None, :, None, :]
        r = (b * H + h) * Nb + i
        blocks = [int(c) for c in col_idx[row_ptr[r]:row_ptr[r + 1]]]
        out[(b, h, i)] = attend_rows(qd[b:b + 1, :, hi:hi + 1, :], kd[b:b + 1, :, hi:hi + 1, :],
                                     vf, 0, 0, i, blocks, scale, block)
    return out
