"""The Ulysses head-sharded wrapper (block_sparse_attention_sa_gb300.ulysses).

CPU tests run real gloo ranks (world sizes 2 and 3, uneven sequence shards):
the re-layout is exact and invertible, each rank receives exactly its heads
of the whole sequence, and a layer run on head shards (with the oracle as the
per-rank attention, since these ranks have no GPU) gives every rank exactly
its token range of the single-rank oracle's output. The GPU test checks that
the wrapper on one rank is the plain library call, bit for bit.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spawn(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return sorted(res, key=lambda d: d["rank"])


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    return dist


def _relayout_main(rank, world, port, out, S, H, dtype):
    dist = _init(rank, world, port)
    try:
        from block_sparse_attention_sa_gb300 import ulysses as U
        g = torch.Generator().manual_seed(7)
        full = torch.randn((2, S, H, 16), generator=g).to(dtype)   # the same on every rank
        s, e = U.shard_bounds(S, world)[rank]
        Hn = H // world
        heads = U.seq_to_heads(full[:, s:e].contiguous(), S)
        back = U.heads_to_seq(heads, e - s)
        lse_full = torch.randn((2, H, S), generator=g)
        lse_back = U.lse_heads_to_seq(lse_full[:, rank * Hn:(rank + 1) * Hn].contiguous(), e - s)
        out.put({"rank": rank,
                 "heads_exact": bool(torch.equal(heads, full[:, :, rank * Hn:(rank + 1) * Hn])),
                 "roundtrip_exact": bool(torch.equal(back, full[:, s:e])),
                 "lse_exact": bool(torch.equal(lse_back, lse_full[:, :, s:e]))})
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,S,H,dtype", [(2, 1000, 4, torch.bfloat16), (3, 1000, 6, torch.float32),
                                             (2, 64, 2, torch.float64)])
def test_relayout_is_exact_and_invertible(world, S, H, dtype):
    for r in _spawn(_relayout_main, world, S, H, dtype):
        assert r["heads_exact"] and r["roundtrip_exact"] and r["lse_exact"], r


def _oracle_layer_main(rank, world, port, out):
    dist = _init(rank, world, port)
    try:
        import oracle
        import sa_inputs
        from block_sparse_attention_sa_gb300 import ulysses as U
        cfg, q, k, v = sa_inputs.make_inputs("tiny")          # S = 1024, H = 4
        tau = float(np.float32(cfg.tau))
        s, e = U.shard_bounds(cfg.S, world)[rank]

        def attend(qh, kh, vh):
            # the per-rank layer on a head shard: the oracle stands in for the
            # library here (these ranks have no GPU)
            ref = oracle.route_ref(qh, kh, cfg.P, tau)
            o, lse = oracle.attn_ref(qh, kh, vh, ref["row_ptr"], ref["col_idx"])
            return torch.from_numpy(o), torch.from_numpy(lse)

        o, lse = U.ulysses_attention(q[:, s:e].contiguous(), k[:, s:e].contiguous(),
                                     v[:, s:e].contiguous(), cfg.S, attend)
        ref = oracle.route_ref(q, k, cfg.P, tau)
        o_full, lse_full = oracle.attn_ref(q, k, v, ref["row_ptr"], ref["col_idx"])
        out.put({"rank": rank, "o_exact": bool(np.array_equal(o.numpy(), o_full[:, s:e])),
                 "lse_exact": bool(np.array_equal(lse.numpy(), lse_full[:, :, s:e]))})
    finally:
        dist.destroy_process_group()


def test_head_sharded_layer_equals_the_single_rank_layer():
    for r in _spawn(_oracle_layer_main, 2):
        assert r["o_exact"] and r["lse_exact"], r


def test_shard_bounds_cover_the_sequence_once():
    from block_sparse_attention_sa_gb300 import ulysses as U
    for S, N in ((38247, 4), (1024, 2), (7, 3)):
        b = U.shard_bounds(S, N)
        assert b[0][0] == 0 and b[-1][1] == S
        assert all(b[i][1] == b[i + 1][0] for i in range(N - 1))
        assert max(e - s for s, e in b) - min(e - s for s, e in b) <= 1


@pytest.mark.gpu
def test_one_rank_is_the_plain_library_call():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import lib
    import sa_inputs
    sa = lib()
    from block_sparse_attention_sa_gb300 import ulysses as U
    cfg, q, k, v = sa_inputs.make_inputs("mid")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1 = U.ulysses_layer(qd, kd, vd, cfg.S, cfg.P, cfg.tau, dev_status=st)
    rp, ci = sa.sa_route(qd, kd, cfg.P, cfg.tau, dev_status=st)
    o2, l2 = sa.sa_attn_sparse(qd, kd, vd, rp, ci, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
