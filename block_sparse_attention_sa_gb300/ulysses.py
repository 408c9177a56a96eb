"""Ulysses head-sharded execution of the routed attention layer across ranks.

The pages run the layer under Ulysses sequence parallelism on four GPUs
("Making MiniMax-H3 up to 9x faster on H100s", section "The setup"; the
Sol-Engine H3-DataCenter release page, "Distributed execution" row of its
table): every rank holds a contiguous range of the packed sequence with all
heads. Routing and attention are independent per head, so an all-to-all turns
that layout into every token of H/N heads, each rank routes and attends its
heads over the whole sequence, and the inverse all-to-all returns each rank's
token range with all heads.

This module is plumbing around the library's calls: the two all-to-alls
(torch.distributed: NCCL on GPUs, gloo on CPU) and the per-rank call. It does
no arithmetic of its own. The exchange is outside the kernels: nothing here
gives one rank's kernels another rank's memory.

Layouts (B batch, S tokens in all, H heads, D head dim, N ranks, Hn = H / N):
    sequence-sharded  [B, S_r, H, D]  on rank r, tokens shard_bounds(S, N)[r]
    head-sharded      [B, S, Hn, D]   on rank r, heads [r Hn, (r + 1) Hn)
"""

from __future__ import annotations

from typing import Callable, List, Optional, Tuple

import torch
import torch.distributed as dist

__all__ = ["shard_bounds", "seq_to_heads", "heads_to_seq", "lse_heads_to_seq",
           "ulysses_attention", "ulysses_layer"]


def _world(group) -> Tuple[int, int]:
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def shard_bounds(S: int, world: int) -> List[Tuple[int, int]]:
    """Rank r's contiguous token range [r S // N, (r + 1) S // N)."""
    return [(r * S // world, (r + 1) * S // world) for r in range(world)]


def _a2a(out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits, group) -> None:
    dist.all_to_all_single(out, inp, output_split_sizes=list(out_splits),
                           input_split_sizes=list(in_splits), group=group)


def seq_to_heads(x: torch.Tensor, S: int, group=None) -> torch.Tensor:
    """[B, S_r, H, D] sequence shard -> [B, S, Hn, D] head shard (all-to-all)."""
    N, rank = _world(group)
    if N == 1:
        return x
    B, S_loc, H, D = x.shape
    if H % N:
        raise ValueError(f"{H} heads do not split over {N} ranks")
    Hn = H // N
    bounds = shard_bounds(S, N)
    if bounds[rank][1] - bounds[rank][0] != S_loc:
        raise ValueError(f"rank {rank} holds {S_loc} tokens, expected {bounds[rank]}")
    # to rank r: heads [r Hn, (r + 1) Hn) of this rank's tokens, as [B, S_loc, Hn, D]
    send = x.reshape(B, S_loc, N, Hn, D).permute(2, 0, 1, 3, 4).contiguous()
    sizes = [B * (e - s) * Hn * D for (s, e) in bounds]
    recv = torch.empty(sum(sizes), dtype=x.dtype, device=x.device)
    _a2a(recv, send.reshape(-1), sizes, [B * S_loc * Hn * D] * N, group)
    parts = recv.split(sizes)
    return torch.cat([p.view(B, e - s, Hn, D) for p, (s, e) in zip(parts, bounds)], dim=1)


def heads_to_seq(y: torch.Tensor, S_loc: int, group=None) -> torch.Tensor:
    """[B, S, Hn, D] head shard -> [B, S_r, H, D] sequence shard (the inverse)."""
    N, rank = _world(group)
    if N == 1:
        return y
    B, S, Hn, D = y.shape
    bounds = shard_bounds(S, N)
    if bounds[rank][1] - bounds[rank][0] != S_loc:
        raise ValueError(f"rank {rank} holds {S_loc} tokens, expected {bounds[rank]}")
    # to rank r: this rank's heads over rank r's tokens
    send = torch.cat([y[:, s:e].reshape(-1) for (s, e) in bounds])
    sizes = [B * (e - s) * Hn * D for (s, e) in bounds]
    recv = torch.empty(B * S_loc * Hn * D * N, dtype=y.dtype, device=y.device)
    _a2a(recv, send, [B * S_loc * Hn * D] * N, sizes, group)
    # from rank r: heads [r Hn, (r + 1) Hn) of this rank's tokens
    return recv.view(N, B, S_loc, Hn, D).permute(1, 2, 0, 3, 4).reshape(B, S_loc, N * Hn, D)


def lse_heads_to_seq(lse: torch.Tensor, S_loc: int, group=None) -> torch.Tensor:
    """[B, Hn, S] log-sum-exp of the head shard -> [B, H, S_r]."""
    N, rank = _world(group)
    if N == 1:
        return lse
    B, Hn, S = lse.shape
    bounds = shard_bounds(S, N)
    send = torch.cat([lse[:, :, s:e].contiguous().reshape(-1) for (s, e) in bounds])
    sizes = [B * Hn * (e - s) for (s, e) in bounds]
    recv = torch.empty(B * Hn * S_loc * N, dtype=lse.dtype, device=lse.device)
    _a2a(recv, send, [B * Hn * S_loc] * N, sizes, group)
    return recv.view(N, B, Hn, S_loc).permute(1, 0, 2, 3).reshape(B, N * Hn, S_loc)


AttendFn = Callable[[torch.Tensor, torch.Tensor, torch.Tensor],
                    Tuple[torch.Tensor, Optional[torch.Tensor]]]


def ulysses_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, S: int,
                      attend: AttendFn, group=None):
    """Sequence shards of Q, K, V -> sequence shard of O (and of the LSE).

    ``attend(q_h, k_h, v_h)`` runs the layer on a head shard [B, S, Hn, D]
    and returns (o_h [B, S, Hn, D], lse_h [B, Hn, S] or None)."""
    S_loc = q.shape[1]
    qh, kh, vh = (seq_to_heads(t, S, group) for t in (q, k, v))
    oh, lseh = attend(qh, kh, vh)
    o = heads_to_seq(oh.contiguous(), S_loc, group)
    lse = None if lseh is None else lse_heads_to_seq(lseh.contiguous(), S_loc, group)
    return o, lse


def ulysses_layer(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, S: int, prefix_len: int,
                  tau: float, group=None, *, mode="threshold", q_block: int = 64,
                  qk_format="bf16", dev_status: Optional[torch.Tensor] = None):
    """One routed attention layer on this rank's sequence shard (CUDA tensors):
    route and attend this rank's heads over the whole sequence with the
    library (sa_route, sa_attn_sparse), between the two all-to-alls."""
    from . import sa_attn_sparse, sa_route

    def attend(qh, kh, vh):
        rp, ci = sa_route(qh, kh, prefix_len, tau, mode=mode, q_block=q_block,
                          dev_status=dev_status)
        return sa_attn_sparse(qh, kh, vh, rp, ci, q_block=q_block, qk_format=qk_format,
                              dev_status=dev_status)

    return ulysses_attention(q, k, v, S, attend, group)
