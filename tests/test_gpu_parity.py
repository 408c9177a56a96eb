"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Routing must give the oracle's kept sets exactly (ties excepted); attention
must match within the tolerances in ``helpers``. Small shapes run in full and
cover the ragged and degenerate cases; the release and long shapes run in the
launch configuration the benchmark times, checked on a seeded sample of
(head, query block) pairs that always includes the first block, the block
holding the end of the prefix, and the ragged tail.
"""

import math

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


def dev(*ts):
    return [t.cuda() for t in ts]


def new_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gpu_route(sa, q, k, P, tau, scale=0.0):
    st = new_status()
    qd, kd = dev(q, k)
    rp, ci = sa.sa_route(qd, kd, P, tau, scale, dev_status=st)
    torch.cuda.synchronize()
    return to_np(rp).astype(np.int64), to_np(ci).astype(np.int64), int(st.item())


def gpu_attn(sa, q, k, v, row_ptr=None, col_idx=None, scale=0.0):
    st = new_status()
    qd, kd, vd = dev(q, k, v)
    if row_ptr is None:
        o, lse = sa.sa_attn_dense(qd, kd, vd, scale, dev_status=st)
    else:
        rp = torch.as_tensor(np.asarray(row_ptr), dtype=torch.int32, device="cuda")
        ci = torch.as_tensor(np.asarray(col_idx), dtype=torch.int32, device="cuda")
        o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, scale, dev_status=st)
    torch.cuda.synchronize()
    return to_np(o), to_np(lse), int(st.item())


def check_route(sa, q, k, P, tau, scale=0.0):
    B, S, H, D = q.shape
    Nb = oracle.num_blocks(S)
    ref = oracle.route_ref(q, k, P, f32(tau), scale=f32(scale) if scale else None)
    rp, ci, st = gpu_route(sa, q, k, P, tau, scale)
    assert st == 0, f"device status {st:#x}"
    assert rp[-1] <= len(ci)
    bad, ties = compare_route(rp, ci[:rp[-1]], ref, B, H, Nb)
    assert bad == 0, f"{bad} routing decisions differ outside ties ({ties} ties)"
    return ref, rp, ci


def check_attn_full(sa, q, k, v, rp, ci, scale=0.0):
    o, lse, st = gpu_attn(sa, q, k, v, rp, ci, scale)
    assert st == 0, f"device status {st:#x}"
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci, scale=f32(scale) if scale else None)
    l2, mx, l2_64 = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx, l2_64)
    assert lse_ok(lse, lse_ref)
    return o, lse


# ------------------------------------------------------------ small shapes --

SMALL = [  # (S, H, D, P, tau)
    (1, 2, 64, 0, 1.0),
    (50, 2, 128, 50, 1.0),
    (64, 3, 64, 1, 1.0),
    (65, 2, 128, 0, 1.0),
    (130, 2, 64, 64, 1.0),
    (200, 1, 128, 0, 0.0),
    (383, 2, 128, 100, 1.0),
    (640, 2, 64, 0, 1.5),
    (1000, 2, 128, 951, 1.0),
]


@pytest.mark.parametrize("S,H,D,P,tau", SMALL)
def test_small_shapes_route_and_attention(sa, S, H, D, P, tau):
    q, k, v = sa_inputs.random_small(S, H, D, seed=S + H + D)
    ref, rp, ci = check_route(sa, q, k, P, tau)
    check_attn_full(sa, q, k, v, ref["row_ptr"], ref["col_idx"])


def test_dense_small_against_dense_oracle(sa):
    q, k, v = sa_inputs.random_small(333, 3, 128, seed=21)
    o, lse, st = gpu_attn(sa, q, k, v)
    assert st == 0
    o_ref, lse_ref = oracle.attn_dense_ref(q, k, v)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(lse, lse_ref)


def test_custom_softmax_scale(sa):
    q, k, v = sa_inputs.random_small(300, 2, 64, seed=4)
    ref, rp, ci = check_route(sa, q, k, 64, 1.0, scale=0.3)
    check_attn_full(sa, q, k, v, ref["row_ptr"], ref["col_idx"], scale=0.3)


def test_batch_and_strided_views(sa):
    # B = 2, heads 1..3 of a 5-head buffer: non-contiguous b/s/h strides
    g = torch.Generator().manual_seed(8)
    big = [torch.randn((2, 300, 5, 128), generator=g).to(torch.bfloat16) for _ in range(3)]
    q, k, v = (t[:, :, 1:4, :] for t in big)
    ref = oracle.route_ref(q, k, 70, 1.0)
    qd, kd, vd = (t.cuda()[:, :, 1:4, :] for t in big)
    assert not qd.is_contiguous()
    st = new_status()
    rp, ci = sa.sa_route(qd, kd, 70, 1.0, dev_status=st)
    o = torch.empty((2, 300, 3, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, o=o, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rpn, cin = to_np(rp).astype(np.int64), to_np(ci).astype(np.int64)
    bad, _ = compare_route(rpn, cin[:rpn[-1]], ref, 2, 3, 5)
    assert bad == 0
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rpn, cin)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(to_np(lse), lse_ref)


def test_empty_rows_give_zero_output_and_neg_inf_lse(sa):
    S, H, D = 256, 1, 64
    q, k, v = sa_inputs.random_small(S, H, D, seed=30)
    rows = [[0, 2], [], [1, 2, 3], []]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    ci = np.array([j for r in rows for j in r])
    o, lse, st = gpu_attn(sa, q, k, v, rp, ci)
    assert st == 0
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci)
    assert np.all(o[0, 64:128] == 0) and np.all(np.isneginf(lse[0, 0, 64:128]))
    assert np.all(o[0, 192:256] == 0) and np.all(np.isneginf(lse[0, 0, 192:256]))
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(lse, lse_ref)


# ------------------------------------------------------------ Tiny / Mid --

@pytest.fixture(scope="module")
def tiny():
    return sa_inputs.make_inputs("tiny")


@pytest.fixture(scope="module")
def mid():
    return sa_inputs.make_inputs("mid")


def test_tiny_route_bitexact_and_full_attention(sa, tiny):
    cfg, q, k, v = tiny
    ref, rp, ci = check_route(sa, q, k, cfg.P, cfg.tau)
    assert abs(oracle.block_density(ref["kept"]) - 0.25) <= 0.01
    # the attention the CUDA path computes over its own route
    check_attn_full(sa, q, k, v, rp[: len(rp)], ci[: rp[-1]])


def test_mid_route_bitexact_and_full_attention(sa, mid):
    cfg, q, k, v = mid
    ref, rp, ci = check_route(sa, q, k, cfg.P, cfg.tau)
    assert 0.18 <= oracle.block_density(ref["kept"]) <= 0.22
    check_attn_full(sa, q, k, v, ref["row_ptr"], ref["col_idx"])


def test_tau_zero_sparse_equals_dense_bitwise(sa, mid):
    cfg, q, k, v = mid
    rp, ci, st = gpu_route(sa, q, k, cfg.P, 0.0)
    assert st == 0 and rp[-1] == cfg.H * cfg.Nb * cfg.Nb
    o_s, l_s, _ = gpu_attn(sa, q, k, v, rp, ci[: rp[-1]])
    o_d, l_d, _ = gpu_attn(sa, q, k, v)
    assert np.array_equal(o_s, o_d) and np.array_equal(l_s, l_d)


def test_unselected_blocks_are_never_read(sa, mid):
    # perturbing K/V of a key block changes no output row whose route skips it
    cfg, q, k, v = mid
    ref = oracle.route_ref(q, k, cfg.P, f32(cfg.tau))
    rp, ci = ref["row_ptr"], ref["col_idx"]
    o0, l0, _ = gpu_attn(sa, q, k, v, rp, ci)
    h, jstar = 3, 77
    k2, v2 = k.clone(), v.clone()
    k2[0, 64 * jstar:64 * jstar + 64, h] = 7.0
    v2[0, 64 * jstar:64 * jstar + 64, h] = -5.0
    o1, l1, _ = gpu_attn(sa, q, k2, v2, rp, ci)
    kept = ref["kept"][0, h]
    untouched = [i for i in range(cfg.Nb) if not kept[i, jstar]]
    touched = [i for i in range(cfg.Nb) if kept[i, jstar]]
    assert untouched and touched
    for i in untouched:
        sl = slice(64 * i, 64 * i + 64)
        assert np.array_equal(o0[0, sl, h], o1[0, sl, h]), i
        assert np.array_equal(l0[0, h, sl], l1[0, h, sl]), i
    assert any(not np.array_equal(o0[0, 64 * i:64 * i + 64, h], o1[0, 64 * i:64 * i + 64, h])
               for i in touched)
    other = [hh for hh in range(cfg.H) if hh != h]
    assert np.array_equal(o0[:, :, other], o1[:, :, other])


# -------------------------------------------------------- device statuses --

def test_capacity_overflow_is_reported(sa):
    q, k, _ = sa_inputs.random_small(512, 2, 64, seed=2)
    st = new_status()
    col_idx = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    rp, _ = sa.sa_route(q.cuda(), k.cuda(), 0, 0.0, col_idx=col_idx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sa.SA_DEV_CAPACITY
    assert int(rp[-1].item()) == 2 * 8 * 8            # row_ptr stays exact
    assert to_np(col_idx).tolist() == [0, 1, 2, 3, 4]


def test_bad_route_entries_are_reported_and_skipped(sa):
    S, H, D = 256, 1, 64
    q, k, v = sa_inputs.random_small(S, H, D, seed=31)
    rp = np.array([0, 2, 3, 5, 6])
    ci = np.array([0, 9, 1, 2, -3, 3])   # 9 and -3 are outside [0, 4)
    o, lse, st = gpu_attn(sa, q, k, v, rp, ci)
    assert st & sa.SA_DEV_BAD_ROUTE
    good_rp = np.array([0, 1, 2, 3, 4])
    good_ci = np.array([0, 1, 2, 3])
    o_ref, lse_ref = oracle.attn_ref(q, k, v, good_rp, good_ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL


def clean_csr(rp, ci, Nb):
    """The route sa_attn_sparse attends for a CSR that breaks the contract: a
    row whose span is not inside [0, row_ptr[-1]] or is longer than Nb is
    empty; otherwise the row is the set of its entries inside [0, Nb)."""
    nnz = int(rp[-1])
    rows = []
    for r in range(len(rp) - 1):
        beg, end = int(rp[r]), int(rp[r + 1])
        if beg < 0 or end < beg or end - beg > Nb or end > nnz:
            rows.append([])
        else:
            rows.append(sorted({int(j) for j in ci[beg:end] if 0 <= j < Nb}))
    out_rp = np.cumsum([0] + [len(x) for x in rows])
    out_ci = np.array([j for x in rows for j in x], dtype=np.int64)
    return out_rp, out_ci


# Each case breaks the CSR contract in one way; the kernel reports it and
# attends the cleaned route (S = 256: four key blocks).
CORRUPT_CSR = {
    "descending_row": ([0, 3, 4, 5, 6], [2, 1, 0, 1, 2, 3]),
    "duplicate_column": ([0, 3, 4, 5, 6], [0, 1, 1, 1, 2, 3]),
    "decreasing_row_ptr": ([0, 2, 1, 3, 4], [0, 1, 2, 3]),
    "span_past_the_route": ([0, 6, 2, 3, 4], [0, 1, 2, 3]),
}


@pytest.mark.parametrize("case", sorted(CORRUPT_CSR))
def test_corrupt_csr_is_reported_and_the_cleaned_route_attended(sa, case):
    S, H, D = 256, 1, 64
    q, k, v = sa_inputs.random_small(S, H, D, seed=41)
    rp, ci = (np.array(x) for x in CORRUPT_CSR[case])
    o, lse, st = gpu_attn(sa, q, k, v, rp, ci)
    assert st & sa.SA_DEV_BAD_ROUTE
    good_rp, good_ci = clean_csr(rp, ci, 4)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, good_rp, good_ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL
    assert lse_ok(lse, lse_ref)


def test_v_outside_fp16_range_is_reported(sa):
    q, k, v = sa_inputs.random_small(128, 1, 64, seed=3)
    v[0, 5, 0, 3] = 1.0e5
    _, _, st = gpu_attn(sa, q, k, v)
    assert st & sa.SA_DEV_RANGE


def test_forward_host_matches_device_calls(sa):
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    bufs = sa.alloc_layer_buffers(1, cfg.S, cfg.H, cfg.D)
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    o_host = sa.sa_forward_host(qh, kh, vh, cfg.P, cfg.tau, bufs=bufs)
    torch.cuda.synchronize()
    assert int(bufs["status"].item()) == 0
    rp, ci, _ = gpu_route(sa, q, k, cfg.P, cfg.tau)
    o_dev, _, _ = gpu_attn(sa, q, k, v, rp, ci[: rp[-1]])
    assert np.array_equal(to_np(o_host), o_dev)


@pytest.mark.parametrize("B,H,with_lse", [(1, 24, True), (2, 16, False), (2, 16, True), (1, 56, True)])
def test_forward_host_head_groups_match_device_calls(sa, B, H, with_lse):
    # H >= 16 splits the layer into head groups whose copies overlap compute;
    # the result must be the one-call result bit for bit (the route and the
    # tile pairing are per head)
    S, D, P, tau = 1000, 128, 100, 1.0
    qs, ks, vs = zip(*(sa_inputs.random_small(S, H, D, seed=40 + b) for b in range(B)))
    q, k, v = (torch.cat(t, dim=0) for t in (qs, ks, vs))
    bufs = sa.alloc_layer_buffers(B, S, H, D)
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    lse_host = torch.empty((B, H, S), dtype=torch.float32).pin_memory() if with_lse else None
    o_host = sa.sa_forward_host(qh, kh, vh, P, tau, bufs=bufs, lse_host=lse_host)
    torch.cuda.synchronize()
    assert int(bufs["status"].item()) == 0
    rp, ci, _ = gpu_route(sa, q, k, P, tau)
    o_dev, lse_dev, _ = gpu_attn(sa, q, k, v, rp, ci[: rp[-1]])
    assert np.array_equal(to_np(o_host), o_dev)
    if with_lse:
        assert np.array_equal(to_np(lse_host), lse_dev)


# --------------------------------------------- release / dense / long shapes --

@pytest.fixture(scope="module")
def release():
    cfg, q, k, v = sa_inputs.make_inputs("release")
    return cfg, q, k, v


def _sampled_attention_check(sa, cfg, q, k, v, rp, ci, seed, dense=False):
    qd, kd, vd = dev(q, k, v)
    st = new_status()
    if dense:
        o, lse = sa.sa_attn_dense(qd, kd, vd, dev_status=st)
    else:
        rpd = torch.as_tensor(rp, dtype=torch.int32, device="cuda")
        cid = torch.as_tensor(ci, dtype=torch.int32, device="cuda")
        o, lse = sa.sa_attn_sparse(qd, kd, vd, rpd, cid, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Nb, n_sink = cfg.Nb, (cfg.P + 63) // 64
    items = sample_items(1, cfg.H, Nb, 8, 16, seed, must=(0, n_sink - 1, Nb - 2, Nb - 1))
    if dense:
        ref = oracle.attn_dense_ref(q, k, v, items=items)
    else:
        ref = oracle.attn_ref(q, k, v, rp, ci, items=items)
    o_np = o.float().cpu().double().numpy()
    lse_np = lse.cpu().double().numpy()
    og, lg = gather_rows(o_np, lse_np, items, cfg.S)
    orf, lrf = ref_rows(ref, items)
    l2, mx, l2_64 = out_errors(og, orf)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx, l2_64)
    assert lse_ok(lg, lrf)


@pytest.mark.parametrize("S,H", [(341 * 64, 3), (256 * 64, 4), (205 * 64, 5), (683 * 64 - 7, 3)])
def test_route_row_counts_around_the_scan_passes(sa, S, H):
    # row_ptr is a scan over the route's H * Nb rows taken 1024 rows per pass:
    # 1023, 1024, 1025 and 2049 rows put the last pass just short of, exactly
    # at and just past a pass boundary; the CSR must be well formed and
    # encode the oracle's route in every row (outside the tie window)
    q, k, _ = sa_inputs.random_small(S, H, 64, seed=S + H)
    Nb = oracle.num_blocks(S)
    assert H * Nb in (1023, 1024, 1025, 2049)
    check_route(sa, q, k, 100, 1.0)


@pytest.mark.parametrize("dense", [False, True])
def test_head_dim_64_with_several_tiles_per_cta(sa, dense):
    # The other D = 64 cases fit in one tile per persistent CTA; here about
    # four tiles run on each (313 key blocks, 157 pairs x 4 heads), so the
    # D = 64 kernel's walks, O reuse and per-tile barrier phases are crossed
    # from tile to tile; the last block is ragged (19 tokens).
    S, H, D, P, tau = 19987, 4, 64, 300, 1.0
    q, k, v = sa_inputs.random_small(S, H, D, seed=64)
    cfg = sa_inputs.Config("d64", S=S, P=P, H=H, D=D, tau=tau, kind="iid")
    assert cfg.Nb == 313
    if dense:
        _sampled_attention_check(sa, cfg, q, k, v, None, None, seed=65, dense=True)
    else:
        ref, rp, ci = check_route(sa, q, k, P, tau)
        _sampled_attention_check(sa, cfg, q, k, v, ref["row_ptr"], ref["col_idx"], seed=66)


def test_release_route_bitexact(sa, release):
    cfg, q, k, v = release
    ref, rp, ci = check_route(sa, q, k, cfg.P, cfg.tau)
    d = oracle.block_density(ref["kept"])
    assert 0.18 <= d <= 0.20, d


def test_release_attention_sampled(sa, release):
    cfg, q, k, v = release
    ref = oracle.route_ref(q, k, cfg.P, f32(cfg.tau))
    _sampled_attention_check(sa, cfg, q, k, v, ref["row_ptr"], ref["col_idx"], seed=1)


def test_dense_release_sampled(sa, release):
    cfg, q, k, v = release
    _sampled_attention_check(sa, cfg, q, k, v, None, None, seed=2, dense=True)


def test_long_route_bitexact_and_attention_sampled(sa):
    cfg, q, k, v = sa_inputs.make_inputs("long")
    ref, rp, ci = check_route(sa, q, k, cfg.P, cfg.tau)
    d = oracle.block_density(ref["kept"])
    assert 0.12 <= d <= 0.15, d
    _sampled_attention_check(sa, cfg, q, k, v, ref["row_ptr"], ref["col_idx"], seed=3)


def test_release_attention_is_deterministic_and_writes_every_row(sa, release):
    # Every tile's work is fixed by the route and the tile list, so repeated
    # calls must agree bit for bit; a race inside the pipeline (a wait that
    # returns early) shows up as a difference here long before a sampled
    # comparison would see it. Outputs start as NaN so an unwritten row shows.
    cfg, q, k, v = release
    qd, kd, vd = dev(q, k, v)
    st = new_status()
    rp, ci = sa.sa_route(qd, kd, cfg.P, cfg.tau, dev_status=st)
    outs = []
    for _ in range(3):
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((1, cfg.H, cfg.S), float("nan"), device="cuda")
        sa.sa_attn_sparse(qd, kd, vd, rp, ci, o=o, lse=lse, dev_status=st)
        torch.cuda.synchronize()
        outs.append((o, lse))
    assert int(st.item()) == 0
    o0, l0 = outs[0]
    assert not torch.isnan(o0).any() and not torch.isnan(l0).any()
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), l0.view(torch.int32))


@pytest.mark.parametrize("S", [4096 * 64, 4096 * 64 - 17])
def test_largest_supported_sequence(sa, S):
    # 4096 key blocks is the most one attention tile's walk can list
    # (kMaxNbAttn); the planner's shared-memory walk buffers are full here.
    H, D, P, tau = 1, 128, 951, 1.2
    q, k, v = sa_inputs.random_small(S, H, D, seed=5)
    ref, rp, ci = check_route(sa, q, k, P, tau)
    Nb = oracle.num_blocks(S)
    assert Nb == 4096
    cfg = sa_inputs.Config("max", S=S, P=P, H=H, D=D, tau=tau, kind="iid")
    _sampled_attention_check(sa, cfg, q, k, v, ref["row_ptr"], ref["col_idx"], seed=6)


def test_bounded_wait_reports_timeout_and_the_context_survives(sa):
    # one warp waits on a barrier nothing completes: the wait gives up after
    # its limit and reports SA_DEV_TIMEOUT, and later work runs normally
    L = sa.load_library()
    st = new_status()
    assert L.sa_check_wait_timeout(st.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(st.item()) & sa.SA_DEV_TIMEOUT
    assert L.sa_dev_status_decode(int(st.item())) == 5          # SA_ERR_TIMEOUT
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    ref, rp, ci = check_route(sa, q, k, cfg.P, cfg.tau)
    check_attn_full(sa, q, k, v, rp, ci[:rp[-1]])


def test_a_timeout_left_in_the_status_word_does_not_abort_later_calls(sa):
    # the status word accumulates bits across calls: after a timeout was
    # reported into it, later calls that share it still run to completion
    L = sa.load_library()
    st = new_status()
    assert L.sa_check_wait_timeout(st.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(st.item()) & sa.SA_DEV_TIMEOUT
    cfg, q, k, v = sa_inputs.make_inputs("mid")
    qd, kd, vd = dev(q, k, v)
    rp, ci = sa.sa_route(qd, kd, cfg.P, cfg.tau, dev_status=st)
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == sa.SA_DEV_TIMEOUT          # nothing new was reported
    rp_n = to_np(rp).astype(np.int64)
    ci_n = to_np(ci).astype(np.int64)[: rp_n[-1]]
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp_n, ci_n)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL
    assert lse_ok(to_np(lse), lse_ref)


@pytest.mark.parametrize("name,q_block", [("tiny", 64), ("mid", 64), ("mid", 128)])
def test_prepare_then_run_equals_attn_sparse(sa, name, q_block):
    # sa_attn_sparse in its two halves, other work enqueued in between: the
    # same output bit for bit
    cfg, q, k, v = sa_inputs.make_inputs(name)
    qd, kd, vd = dev(q, k, v)
    st = new_status()
    rp, ci = sa.sa_route(qd, kd, cfg.P, cfg.tau, q_block=q_block, dev_status=st)
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, q_block=q_block, dev_status=st)
    p = sa.make_params(qd, kd, vd, o, q_block=q_block)
    ws = torch.empty(sa.sa_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    sa.sa_attn_prepare(vd, rp, ci, workspace=ws, q_block=q_block, dev_status=st)
    junk = torch.randn(1 << 20, device="cuda").sum()        # unrelated work in between
    o2, lse2 = sa.sa_attn_run(qd, kd, rp, ci, workspace=ws, v_like=vd, q_block=q_block,
                              dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.isfinite(junk)
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
