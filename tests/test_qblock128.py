"""GPU parity of the router with 128-token query blocks (sa_params.q_block).

With q_block = 128 the router pools each 128-token query block, scores it
against every 64-token key block and forces the two key blocks inside it; the
CSR still has one row per 64-token block, rows 2i and 2i + 1 holding query
block i's list. Attention with q_block = 128 takes the 128-token query blocks
as its tiles (no pairing step). Checked like the default route: kept sets
equal to the oracle's outside its ties, attention within the tolerances of
``helpers``, on ragged and degenerate shapes, the tiny and mid workloads in
full and the release workload in the launch configuration the benchmark
times (route in full, attention on a seeded sample).
"""

import numpy as np
import pytest
import torch

import oracle
import sa_inputs
from helpers import (L2_TOL, MAXABS_TOL, compare_route, f32, gather_rows, lib, lse_ok,
                     out_errors, ref_rows, sample_items, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


def route_both(sa, q, k, P, tau, mode="threshold"):
    B, S, H, D = q.shape
    Nb = oracle.num_blocks(S)
    ref = oracle.route_ref(q, k, P, f32(tau), mode=mode, q_block=128)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rp, ci = sa.sa_route(q.cuda(), k.cuda(), P, tau, mode=mode, q_block=128, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rp, ci = to_np(rp).astype(np.int64), to_np(ci).astype(np.int64)
    ci = ci[:rp[-1]]
    bad, ties = compare_route(rp, ci, ref, B, H, Nb)
    assert bad == 0, f"{bad} decisions differ outside ties ({ties} ties)"
    # both 64-token rows of a query block carry the same list
    for bh in range(B * H):
        for i in range(0, Nb - 1, 2):
            r = bh * Nb + i
            assert np.array_equal(ci[rp[r]:rp[r + 1]], ci[rp[r + 1]:rp[r + 2]]), r
    return ref, rp, ci


def attn_check(sa, q, k, v, rp, ci, q_block=128):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rpd = torch.as_tensor(rp, dtype=torch.int32, device="cuda")
    cid = torch.as_tensor(ci, dtype=torch.int32, device="cuda")
    o, lse = sa.sa_attn_sparse(q.cuda(), k.cuda(), v.cuda(), rpd, cid, q_block=q_block,
                               dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(to_np(lse), lse_ref)


SMALL = [  # (S, H, D, P, tau): S = 1 and 65 (one query block), odd and even Nb, ragged tails
    (1, 2, 64, 0, 1.0),
    (65, 2, 128, 0, 0.5),
    (127, 1, 64, 64, 1.0),
    (383, 2, 128, 100, 0.7),
    (640, 2, 64, 0, 0.0),
    (700, 2, 64, 130, 1.0),
    (1000, 2, 128, 951, 0.3),
    (2047, 1, 64, 200, 1.2),
]


@pytest.mark.parametrize("S,H,D,P,tau", SMALL)
def test_small_shapes_route_and_attention(sa, S, H, D, P, tau):
    q, k, v = sa_inputs.random_small(S, H, D, seed=S + 5 * H + D)
    _, rp, ci = route_both(sa, q, k, P, tau)
    attn_check(sa, q, k, v, rp, ci)


@pytest.mark.parametrize("mode,tau", [("dense_prefix_queries", 1.0), ("top_mass", 0.5),
                                      ("top_mass", 0.9)])
@pytest.mark.parametrize("S,P", [(383, 100), (1000, 130), (2047, 951)])
def test_other_modes_small(sa, mode, tau, S, P):
    q, k, v = sa_inputs.random_small(S, 2, 64, seed=S + 3)
    ref, rp, ci = route_both(sa, q, k, P, tau, mode)
    if mode == "dense_prefix_queries":
        n_rows = 2 * ((P + 127) // 128)
        assert ref["kept"][:, :, :n_rows].all()
    attn_check(sa, q, k, v, rp, ci)


def test_square_route_through_neighbour_tiles_is_exact(sa):
    # q_block = 128 only fixes the attention tiles; a CSR whose two halves
    # differ is still attended exactly (the other half's blocks are masked).
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    ref = oracle.route_ref(q, k, cfg.P, f32(cfg.tau))
    attn_check(sa, q, k, v, ref["row_ptr"], ref["col_idx"], q_block=128)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_tiny_and_mid_route_and_full_attention(sa, name):
    cfg, q, k, v = sa_inputs.make_inputs(name)
    _, rp, ci = route_both(sa, q, k, cfg.P, cfg.tau)
    attn_check(sa, q, k, v, rp, ci)


def test_release_route_bitexact_and_attention_sampled(sa):
    cfg, q, k, v = sa_inputs.make_inputs("release")
    ref, rp, ci = route_both(sa, q, k, cfg.P, cfg.tau)
    d = oracle.block_density(ref["kept"])
    assert 0.1 < d < 0.3, d
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rpd = torch.as_tensor(rp, dtype=torch.int32, device="cuda")
    cid = torch.as_tensor(ci, dtype=torch.int32, device="cuda")
    o = torch.full_like(qd, float("nan"))
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rpd, cid, o=o, q_block=128, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert not torch.isnan(o).any()
    Nb, n_sink = cfg.Nb, (cfg.P + 63) // 64
    items = sample_items(1, cfg.H, Nb, 8, 16, seed=4, must=(0, n_sink - 1, Nb - 2, Nb - 1))
    refo = oracle.attn_ref(q, k, v, rp, ci, items=items)
    og, lg = gather_rows(to_np(o), to_np(lse), items, cfg.S)
    orf, lrf = ref_rows(refo, items)
    l2, mx, _ = out_errors(og, orf)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(lg, lrf)


def test_batch_and_strided_views(sa):
    # B = 2, heads 1..3 of a 5-head buffer, a ragged S: non-contiguous b/s/h strides
    g = torch.Generator().manual_seed(12)
    big = [torch.randn((2, 333, 5, 64), generator=g).to(torch.bfloat16) for _ in range(3)]
    q, k, v = (t[:, :, 1:4, :] for t in big)
    qd, kd, vd = (t.cuda()[:, :, 1:4, :] for t in big)
    assert not qd.is_contiguous()
    ref = oracle.route_ref(q, k, 70, f32(0.9), q_block=128)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rp, ci = sa.sa_route(qd, kd, 70, 0.9, q_block=128, dev_status=st)
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, q_block=128, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rpn, cin = to_np(rp).astype(np.int64), to_np(ci).astype(np.int64)
    bad, _ = compare_route(rpn, cin[:rpn[-1]], ref, 2, 3, oracle.num_blocks(333))
    assert bad == 0
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rpn, cin)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(to_np(lse), lse_ref)


def test_forward_host_matches_device_calls(sa):
    # the whole layer from pinned host memory, in head groups, with 128-token
    # query blocks: bit for bit the result of the two device calls
    B, S, H, D, P, tau = 1, 1000, 24, 128, 100, 1.0
    q, k, v = sa_inputs.random_small(S, H, D, seed=77)
    bufs = sa.alloc_layer_buffers(B, S, H, D)
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    lse_host = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    o_host = sa.sa_forward_host(qh, kh, vh, P, tau, bufs=bufs, q_block=128, lse_host=lse_host)
    torch.cuda.synchronize()
    assert int(bufs["status"].item()) == 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rp, ci = sa.sa_route(qd, kd, P, tau, q_block=128, dev_status=st)
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, q_block=128, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o_host.view(torch.int16), o.cpu().view(torch.int16))
    assert torch.equal(lse_host.view(torch.int32), lse.cpu().view(torch.int32))
