"""GPU: the tile pairing of sa_attn_sparse.

Each 128-row attention tile holds two 64-row query blocks and walks the union
of their key lists, so sa_attn_sparse first pairs the query blocks of every
head: greedily, heaviest edge first, where an edge's weight is the number of
key blocks the two lists share, among blocks at most W apart; ties go to the
neighbour pair (2p, 2p+1), then to a fixed hash of the edge; blocks left
without a candidate pair up in index order. The tests read the
tile list the call leaves at the end of its workspace and compare it with
that greedy matching written out plainly below, then check the attention
itself against the oracle on a route whose best partners are not neighbours.
"""

import numpy as np
import pytest
import torch

import oracle
import sa_inputs
from helpers import L2_TOL, MAXABS_TOL, lib, lse_ok, out_errors, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


W = 32   # candidates: blocks at most 32 apart


def edge_hash(x):
    m = 0xFFFFFFFF
    x = (x * 0x9E3779B1) & m
    x ^= x >> 15
    x = (x * 0x2C1B3C6D) & m
    x ^= x >> 12
    return x


def greedy_pairs(row_ptr, col_idx, nb, w):
    """The tile list of one head: sorted (a, b) with a < b, b = -1 for a lone block."""
    sets = [set(col_idx[row_ptr[i]:row_ptr[i + 1]].tolist()) for i in range(nb)]
    edges = []
    for a in range(nb):
        for b in range(a + 1, min(nb, a + w + 1)):
            d = b - a
            key = (len(sets[a] & sets[b]), int(d == 1 and a % 2 == 0), edge_hash(a * 128 + d) >> 8,
                   d, a)
            edges.append((key, a, b))
    edges.sort(reverse=True)
    mate = [-1] * nb
    for _, a, b in edges:
        if mate[a] < 0 and mate[b] < 0:
            mate[a], mate[b] = b, a
    left = [u for u in range(nb) if mate[u] < 0]
    for x in range(0, len(left) - 1, 2):
        mate[left[x]], mate[left[x + 1]] = left[x + 1], left[x]
    return [(u, mate[u]) for u in range(nb) if mate[u] < 0 or u < mate[u]]


def run_sparse(sa, q, k, v, rp, ci):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rpd = torch.as_tensor(np.asarray(rp), dtype=torch.int32, device="cuda")
    cid = torch.as_tensor(np.asarray(ci), dtype=torch.int32, device="cuda")
    p = sa.make_params(qd, kd, vd, qd)
    nbytes = sa.sa_attn_workspace_bytes(p)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rpd, cid, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    B, S, H, _ = q.shape
    nb = oracle.num_blocks(S)
    n_pairs = (nb + 1) // 2
    list_bytes = (B * H * n_pairs * 4 + 255) // 256 * 256
    raw = to_np(ws[nbytes - list_bytes:nbytes - list_bytes + B * H * n_pairs * 4].clone())
    tiles = raw.view(np.uint32).reshape(B * H, n_pairs)
    return to_np(o), to_np(lse), int(st.item()), tiles


def decode(tiles_row):
    return [(int(t & 0xFFFF), -1 if (t >> 16) == 0xFFFF else int(t >> 16)) for t in tiles_row]


def check_tiles(tiles, rp, ci, B, H, nb):
    for bh in range(B * H):
        r0 = bh * nb
        rows = np.asarray(rp[r0:r0 + nb + 1]) - rp[r0]
        cols = np.asarray(ci[rp[r0]:rp[r0 + nb]])
        assert decode(tiles[bh]) == greedy_pairs(rows, cols, nb, W), bh


def test_tiny_route_pairs_are_the_greedy_matching(sa):
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    rp, ci = sa.sa_route(q.cuda(), k.cuda(), cfg.P, cfg.tau)
    rp, ci = to_np(rp).astype(np.int64), to_np(ci).astype(np.int64)
    ci = ci[: rp[-1]]
    o, lse, st, tiles = run_sparse(sa, q, k, v, rp, ci)
    assert st == 0
    check_tiles(tiles, rp, ci, 1, cfg.H, cfg.Nb)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(lse, lse_ref)


def test_mid_route_pairs_are_the_greedy_matching(sa):
    cfg, q, k, v = sa_inputs.make_inputs("mid")
    ref = oracle.route_ref(q, k, cfg.P, float(np.float32(cfg.tau)))
    rp, ci = ref["row_ptr"], ref["col_idx"]
    _, _, st, tiles = run_sparse(sa, q, k, v, rp, ci)
    assert st == 0
    check_tiles(tiles, rp, ci, 1, cfg.H, cfg.Nb)   # Nb = 128 > 2W + 1: windowed candidates


def far_partner_route(nb, period, seed):
    """Rows i and i + period share a list; neighbours share only the forced blocks."""
    rng = np.random.default_rng(seed)
    base = [sorted(set(rng.choice(nb, size=nb // 4, replace=False).tolist())) for _ in range(period)]
    rows = []
    for i in range(nb):
        rows.append(sorted(set(base[i % period]) | {0, i}))
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    return rp, np.array([j for r in rows for j in r])


@pytest.mark.parametrize("S,H,D,period", [(1000, 2, 128, 5), (2047, 1, 64, 7)])
def test_far_partners_pair_up_and_attention_matches(sa, S, H, D, period):
    q, k, v = sa_inputs.random_small(S, H, D, seed=S + period)
    nb = oracle.num_blocks(S)
    rps, cis = [], []
    off = 0
    for h in range(H):
        rp, ci = far_partner_route(nb, period, seed=h)
        rps.append(rp[:-1] + off)
        cis.append(ci)
        off += len(ci)
    rp = np.concatenate(rps + [[off]])
    ci = np.concatenate(cis)
    o, lse, st, tiles = run_sparse(sa, q, k, v, rp, ci)
    assert st == 0
    check_tiles(tiles, rp, ci, 1, H, nb)
    for bh in range(H):   # blocks sharing a list pair up (all but a few lone ones)
        far = sum(1 for a, b in decode(tiles[bh]) if b >= 0 and (b - a) % period == 0)
        assert far >= nb // 2 - period
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(lse, lse_ref)
