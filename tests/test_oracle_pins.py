"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one step of the oracle to a closed form, a hand-worked
example, a brute-force loop or an invariant, chosen so that a plausible slip
(a dropped term, a wrong sign or axis, a transposed operand, dividing a
partial block by 64) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import sa_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# ---------------------------------------------------------------- pooling --

def test_pool_ragged_tail_closed_form():
    # token t of head h, dim d holds t + 100 h + d (all exact in bf16 up to 256)
    S, H, D = 70, 2, 3
    x = np.zeros((1, S, H, D))
    for t in range(S):
        for h in range(H):
            for d in range(D):
                x[0, t, h, d] = t + 100 * h + d
    pooled = oracle.pool_blocks(x)
    assert pooled.shape == (1, H, 2, D)
    for h in range(H):
        for d in range(D):
            assert pooled[0, h, 0, d] == 31.5 + 100 * h + d     # mean of 0..63
            assert pooled[0, h, 1, d] == 66.5 + 100 * h + d     # mean of 64..69 (6 tokens)


def test_block_bounds():
    starts, counts = oracle.block_bounds(38247)
    assert len(starts) == 598 and counts[-1] == 39 and counts[:-1].min() == 64
    starts, counts = oracle.block_bounds(64)
    assert list(counts) == [64]
    assert oracle.num_blocks(112640) == 1760


# ----------------------------------------------------------------- router --

def test_pooled_logits_hand_example():
    qbar = np.array([[[[1.0, 2.0], [0.0, -1.0]]]])      # [1,1,2,2]
    kbar = np.array([[[[3.0, 0.5], [-2.0, 4.0], [1.0, 1.0]]]])  # [1,1,3,2]
    s = oracle.pooled_logits(qbar, kbar, 0.5)
    want = np.array([[4.0 * 0.5, 6.0 * 0.5, 3.0 * 0.5],
                     [-0.5 * 0.5, -4.0 * 0.5, -1.0 * 0.5]])
    np.testing.assert_array_equal(s[0, 0], want)


def test_softmax_closed_form():
    s = np.log(np.array([[1.0, 2.0, 3.0, 6.0]]))
    p = oracle.pooled_softmax(s)
    np.testing.assert_allclose(p, [[1 / 12, 2 / 12, 3 / 12, 6 / 12]], rtol=1e-15)
    # shift invariance of the max-subtracted form, with huge logits
    p2 = oracle.pooled_softmax(s + 1000.0)
    np.testing.assert_allclose(p2, p, rtol=1e-13)


def _hand_inputs(spec):
    S, H, D = spec["S"], spec["H"], spec["D"]
    q = np.zeros((1, S, H, D), np.float32)
    k = np.zeros((1, S, H, D), np.float32)
    q[0, :, 0, 0] = 1.0
    k[0, 64:128, 0, 0] = 0.5
    k[0, 128:192, 0, 0] = 1.0
    k[0, 192:196, 0, 0] = 4.0      # block 3: 4 tokens of 4 and 4 of 0 -> mean 2
    return bf16(q), bf16(k)


def test_router_hand_worked_fixture():
    spec = json.load(open(os.path.join(GOLDEN, "route_hand_example.json")))
    q, k = _hand_inputs(spec)
    for case in spec["cases"]:
        r = oracle.route_ref(q, k, spec["prefix_len"], case["tau"], scale=spec["scale"])
        rp, ci = r["row_ptr"], r["col_idx"]
        rows = [list(ci[rp[i]:rp[i + 1]]) for i in range(len(rp) - 1)]
        assert rows == case["rows"], (case["tau"], rows)


def test_threshold_is_inclusive_at_exact_uniform_share():
    # identical key blocks -> every pooled probability is exactly 1/Nb
    S, H, D = 256, 1, 4
    q = bf16(np.random.default_rng(0).standard_normal((1, S, H, D)))
    k = bf16(np.ones((1, S, H, D)))
    Nb = 4
    r = oracle.route_ref(q, k, 0, 1.0)
    np.testing.assert_array_equal(r["p"], np.full((1, 1, Nb, Nb), 1.0 / Nb))
    assert r["kept"].all()                                  # p >= tau/Nb with equality
    assert oracle.route_ref(q, k, 0, 0.999)["kept"].all()
    only_forced = oracle.route_ref(q, k, 0, 1.001)["kept"][0, 0]
    np.testing.assert_array_equal(only_forced, np.eye(Nb, dtype=bool))


def test_sink_blocks_and_diagonal_are_forced():
    f = oracle.forced_mask(5, 65)          # P = 65 touches blocks 0 and 1
    assert f[:, :2].all() and not f[0, 2:].any()
    assert np.diag(f).all()
    f0 = oracle.forced_mask(5, 0)          # no prefix: only the diagonal
    np.testing.assert_array_equal(f0, np.eye(5, dtype=bool))
    f64 = oracle.forced_mask(5, 64)        # exactly one full block
    assert f64[:, 0].all() and not f64[0, 1:].any()


@pytest.fixture(scope="module")
def tiny_route():
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    return cfg, q, k, v, oracle.route_ref(q, k, cfg.P, cfg.tau)


def test_route_invariants_tiny(tiny_route):
    cfg, q, k, v, r = tiny_route
    rp, ci = r["row_ptr"], r["col_idx"]
    Nb = cfg.Nb
    n_sink = (cfg.P + 63) // 64
    for row in range(cfg.H * Nb):
        cols = ci[rp[row]:rp[row + 1]]
        assert np.all(np.diff(cols) > 0)                   # sorted, unique
        i = row % Nb
        assert i in cols                                    # diagonal
        assert all(j in cols for j in range(n_sink))        # sink
    # density the Tiny config is calibrated to
    assert abs(oracle.block_density(r["kept"]) - 0.25) <= 0.01


def test_route_monotone_in_tau(tiny_route):
    cfg, q, k, v, _ = tiny_route
    prev = None
    for tau in (0.0, 0.9, 1.0, 1.01, 1.02, 1.1, 3.0):
        kept = oracle.route_ref(q, k, cfg.P, tau)["kept"]
        if prev is not None:
            assert not (kept & ~prev).any()                # R(tau2) subset of R(tau1)
        prev = kept


def test_tau_zero_keeps_every_block(tiny_route):
    cfg, q, k, v, _ = tiny_route
    assert oracle.route_ref(q, k, cfg.P, 0.0)["kept"].all()


def test_tau_above_max_keeps_only_forced(tiny_route):
    cfg, q, k, v, r = tiny_route
    tau = float(r["p"].max() * cfg.Nb) * 1.0001
    kept = oracle.route_ref(q, k, cfg.P, tau)["kept"]
    forced = oracle.forced_mask(cfg.Nb, cfg.P)
    np.testing.assert_array_equal(kept[0], np.broadcast_to(forced, kept[0].shape))


def test_key_block_permutation_permutes_probabilities(tiny_route):
    cfg, q, k, v, r = tiny_route
    perm = np.random.default_rng(3).permutation(cfg.Nb)
    s = oracle.pooled_logits(r["qbar"], r["kbar"][:, :, perm, :], cfg.scale)
    p_perm = oracle.pooled_softmax(s)
    np.testing.assert_allclose(p_perm, r["p"][..., perm], rtol=1e-12, atol=0)


def test_pooled_route_matches_direct_token_sums():
    # the pooled logit equals the mean over token pairs of scale * q_t . k_u
    q, k, _ = sa_inputs.random_small(130, 1, 8, seed=11)
    r = oracle.route_ref(q, k, 0, 1.0)
    qf, kf = oracle.as_f64(q), oracle.as_f64(k)
    scale = 1 / math.sqrt(8)
    blocks = [(0, 64), (64, 128), (128, 130)]
    s = np.zeros((3, 3))
    for i, (a, b) in enumerate(blocks):
        for j, (c, d) in enumerate(blocks):
            acc = [scale * float(qf[0, t, 0] @ kf[0, u, 0]) for t in range(a, b) for u in range(c, d)]
            s[i, j] = math.fsum(acc) / ((b - a) * (d - c))
    ex = np.exp(s - s.max(axis=1, keepdims=True))
    np.testing.assert_allclose(r["p"][0, 0], ex / ex.sum(axis=1, keepdims=True), rtol=1e-11)


# -------------------------------------------------------------- attention --

def brute_attention(qf, kf, vf, b, h, t, keys, scale):
    """One query token, pure Python: softmax over the listed key tokens."""
    logits = [scale * math.fsum(qf[b, t, h, d] * kf[b, u, h, d] for d in range(qf.shape[3]))
              for u in keys]
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    z = math.fsum(w)
    out = [math.fsum(w[n] * vf[b, u, h, d] for n, u in enumerate(keys)) / z
           for d in range(qf.shape[3])]
    return out, m + math.log(z)


def test_sparse_attention_matches_brute_force_ragged():
    S, H, D = 150, 2, 4            # blocks of 64, 64, 22 tokens
    q, k, v = sa_inputs.random_small(S, H, D, seed=5)
    qf, kf, vf = (oracle.as_f64(x) for x in (q, k, v))
    # hand-chosen route, rows (h, i): includes an empty-looking off-diagonal mix
    rows = {(0, 0): [0, 2], (0, 1): [1], (0, 2): [0, 1, 2],
            (1, 0): [0], (1, 1): [0, 1, 2], (1, 2): [2]}
    Nb = 3
    counts = [len(rows[(h, i)]) for h in range(H) for i in range(Nb)]
    row_ptr = np.concatenate([[0], np.cumsum(counts)])
    col_idx = np.array([j for h in range(H) for i in range(Nb) for j in rows[(h, i)]])
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attn_ref(q, k, v, row_ptr, col_idx)
    for h in range(H):
        for i in range(Nb):
            keys = [u for j in rows[(h, i)] for u in range(64 * j, min(S, 64 * j + 64))]
            for t in range(64 * i, min(S, 64 * i + 64), 7):
                want, want_lse = brute_attention(qf, kf, vf, 0, h, t, keys, scale)
                np.testing.assert_allclose(o[0, t, h], want, rtol=1e-12, atol=1e-14)
                assert abs(lse[0, h, t] - want_lse) < 1e-12


def test_dense_attention_matches_whole_sequence_softmax():
    q, k, v = sa_inputs.random_small(200, 3, 16, seed=7)
    qf, kf, vf = (oracle.as_f64(x) for x in (q, k, v))
    o, lse = oracle.attn_dense_ref(q, k, v)
    for h in range(3):
        s = qf[0, :, h] @ kf[0, :, h].T / 4.0
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        np.testing.assert_allclose(o[0, :, h], (e / e.sum(1, keepdims=True)) @ vf[0, :, h],
                                   rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], (m + np.log(e.sum(1, keepdims=True)))[:, 0],
                                   rtol=1e-13)


def test_tau_zero_sparse_equals_dense(tiny_route):
    cfg, q, k, v, _ = tiny_route
    r0 = oracle.route_ref(q, k, cfg.P, 0.0)
    o_s, l_s = oracle.attn_ref(q, k, v, r0["row_ptr"], r0["col_idx"])
    o_d, l_d = oracle.attn_dense_ref(q, k, v)
    np.testing.assert_allclose(o_s, o_d, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_s, l_d, rtol=0, atol=1e-12)


def test_constant_values_give_constant_output():
    # weights sum to 1 for every row => O == the constant V row
    q, k, _ = sa_inputs.random_small(100, 2, 8, seed=9)
    v = torch.full((1, 100, 2, 8), 0.375, dtype=torch.bfloat16)
    r = oracle.route_ref(q, k, 0, 1.0)
    o, _ = oracle.attn_ref(q, k, v, r["row_ptr"], r["col_idx"])
    np.testing.assert_allclose(o, 0.375, rtol=0, atol=1e-14)


def test_zero_queries_average_the_valid_keys():
    # q = 0 => uniform weights over the valid tokens of the kept blocks;
    # a padded tail that leaked in would shift the mean.
    S, H, D = 100, 1, 4
    q = torch.zeros((1, S, H, D), dtype=torch.bfloat16)
    _, k, v = sa_inputs.random_small(S, H, D, seed=13)
    o, lse = oracle.attn_dense_ref(q, k, v)
    vf = oracle.as_f64(v)
    np.testing.assert_allclose(o[0, 0, 0], vf[0, :, 0].mean(axis=0), rtol=1e-13)
    np.testing.assert_allclose(lse[0, 0], math.log(S), rtol=1e-15)


def test_single_block_sequence_is_dense():
    q, k, v = sa_inputs.random_small(50, 2, 8, seed=17)
    r = oracle.route_ref(q, k, 0, 5.0)
    assert list(r["col_idx"]) == [0, 0]
    o_s, _ = oracle.attn_ref(q, k, v, r["row_ptr"], r["col_idx"])
    o_d, _ = oracle.attn_dense_ref(q, k, v)
    np.testing.assert_array_equal(o_s, o_d)


def test_routed_flops_counts_valid_pairs_only():
    # S = 100: blocks of 64 and 36 tokens; dense route
    rp, ci = oracle.dense_csr(1, 1, 100)
    assert oracle.routed_flops(rp, ci, 1, 1, 100, 8) == 4 * 8 * 100 * 100
    # only the diagonal
    rp = np.array([0, 1, 2]); ci = np.array([0, 1])
    assert oracle.routed_flops(rp, ci, 1, 1, 100, 8) == 4 * 8 * (64 * 64 + 36 * 36)


def test_tie_mask_window():
    ratio = np.array([1.0, 1.0 + 5e-7, 1.0 - 2e-6, 0.5])
    forced = np.array([False, False, False, False])
    np.testing.assert_array_equal(oracle.tie_mask(ratio, forced), [True, True, False, False])


# ------------------------------------------------------------- generators --

def test_generators_shapes_and_determinism():
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    assert q.shape == (1, 1024, 4, 64) and q.dtype == torch.bfloat16
    _, q2, _, _ = sa_inputs.make_inputs("tiny")
    assert torch.equal(q, q2)
    cfg = sa_inputs.get_config("release")
    assert cfg.P + cfg.grid[0] * cfg.grid[1] * cfg.grid[2] == cfg.S
    cfg = sa_inputs.get_config("long")
    assert cfg.S - cfg.P == 110 * 24 * 42 + 809


# ------------------------------------------------- router readings (modes) --

def test_top_mass_hand_example():
    # ranks: 0.5 (block 0), 0.2 (block 1), 0.2 (block 2: equal p, higher index), 0.1
    p = np.array([[0.5, 0.2, 0.2, 0.1]])
    kept, ties = oracle.select_top_mass(p, 0.6)          # 0 < .6, .5 < .6, .7 >= .6
    assert kept[0].tolist() == [True, True, False, False]
    assert ties[0].tolist() == [False, True, True, False]   # equal p across the cut
    kept, ties = oracle.select_top_mass(p, 0.5)          # block 1 has 0.5 above it: not < 0.5
    assert kept[0].tolist() == [True, False, False, False]
    assert ties[0].tolist() == [False, True, False, False]  # its preceding mass equals tau
    kept, _ = oracle.select_top_mass(p, 0.95)
    assert kept[0].tolist() == [True, True, True, True]     # .9 above block 3 is < .95
    kept, _ = oracle.select_top_mass(p, 0.0)
    assert not kept.any()                                   # nothing holds less than 0
    kept, ties = oracle.select_top_mass(np.array([[0.7, 0.3]]), 0.69)
    assert kept[0].tolist() == [True, False] and not ties.any()


def _brute_top_mass(row, tau):
    order = sorted(range(len(row)), key=lambda j: (-row[j], j))
    kept, acc = set(), 0.0
    for j in order:
        if acc < tau:
            kept.add(j)
        acc = math.fsum([acc, row[j]])
    return kept


def test_top_mass_against_brute_force_and_invariants():
    rng = np.random.default_rng(5)
    for trial in range(40):
        n = int(rng.integers(2, 40))
        s = rng.normal(size=n) * float(rng.uniform(0.1, 4.0))
        p = np.exp(s - s.max())
        p /= p.sum()
        tau = float(rng.uniform(0.05, 0.99))
        kept, ties = oracle.select_top_mass(p[None], tau)
        kept, ties = kept[0], ties[0]
        want = _brute_top_mass(p.tolist(), tau)
        got = set(np.nonzero(kept)[0].tolist())
        assert (got ^ want) <= set(np.nonzero(ties)[0].tolist())
        if not ties.any():
            assert got == want
            assert p[kept].sum() >= tau - 1e-12                 # the kept blocks cover tau
            assert p[kept].sum() - p[kept].min() < tau          # and none of them is spare
        kept_hi, _ = oracle.select_top_mass(p[None], min(1.0, tau + 0.05))
        assert not (kept & ~kept_hi[0]).any()                    # monotone in tau
        perm = rng.permutation(n)                                # equivariant if no equal p
        kp, _ = oracle.select_top_mass(p[perm][None], tau)
        if not ties.any():
            assert np.array_equal(kp[0], kept[perm])


def test_route_modes_forced_blocks_and_prefix_rows():
    q, k, _ = sa_inputs.random_small(700, 2, 64, seed=11)
    P = 130                                     # 3 sink blocks
    thr = oracle.route_ref(q, k, P, 1.0)
    dpq = oracle.route_ref(q, k, P, 1.0, mode="dense_prefix_queries")
    top = oracle.route_ref(q, k, P, 0.5, mode="top_mass")
    n_sink, Nb = 3, oracle.num_blocks(700)
    assert dpq["kept"][:, :, :n_sink, :].all()                 # prefix rows keep everything
    assert np.array_equal(dpq["kept"][:, :, n_sink:], thr["kept"][:, :, n_sink:])
    for r in (thr, dpq, top):
        assert r["kept"][..., :n_sink].all()                    # sink columns
        assert r["kept"][..., np.arange(Nb), np.arange(Nb)].all()   # diagonal
        assert not (r["ties"] & r["forced"]).any()
    # top-mass rows cover tau with their unforced-or-forced blocks
    cover = (top["p"] * top["kept"]).sum(-1)
    assert (cover >= 0.5 - 1e-12).all()
    with pytest.raises(ValueError):
        oracle.route_ref(q, k, P, 1.0, mode="z")


# ------------------------------------------- 128-token query blocks ------

def _hand_inputs_qblock128(spec):
    S, H, D = spec["S"], spec["H"], spec["D"]
    q = np.zeros((1, S, H, D), np.float32)
    q[0, 0:64, 0, 0] = 1.0
    q[0, 64:128, 0, 0] = 3.0
    q[0, 192:200, 0, 0] = 9.0      # query block 1: 8 tokens of 9 among 72 -> mean 1
    _, k = _hand_inputs(spec)
    return bf16(q), k


def test_router_qblock128_hand_worked_fixture():
    spec = json.load(open(os.path.join(GOLDEN, "route_hand_example_qblock128.json")))
    q, k = _hand_inputs_qblock128(spec)
    for case in spec["cases"]:
        r = oracle.route_ref(q, k, case["prefix_len"], case["tau"], scale=spec["scale"],
                             q_block=spec["q_block"])
        rp, ci = r["row_ptr"], r["col_idx"]
        rows = [list(ci[rp[i]:rp[i + 1]]) for i in range(len(rp) - 1)]
        assert rows == case["rows"], (case, rows)


def test_pool_qblock128_ragged_tail_closed_form():
    S, H, D = 200, 1, 2
    x = np.zeros((1, S, H, D))
    x[0, :, 0, 0] = np.arange(S)
    x[0, :, 0, 1] = 1.0
    pooled = oracle.pool_blocks(x, 128)
    assert pooled.shape == (1, 1, 2, 2)
    assert pooled[0, 0, 0, 0] == 63.5 and pooled[0, 0, 1, 0] == 163.5   # 72-token tail
    assert (pooled[0, 0, :, 1] == 1.0).all()


def test_qblock128_forced_mask():
    f = oracle.forced_mask(5, 0, q_block=128)       # 5 key blocks -> 3 query blocks
    want = np.array([[1, 1, 0, 0, 0], [0, 0, 1, 1, 0], [0, 0, 0, 0, 1]], dtype=bool)
    np.testing.assert_array_equal(f, want)
    f = oracle.forced_mask(5, 65, q_block=128)      # sink blocks 0 and 1
    assert f[:, :2].all() and f[1, 2:4].all() and f[2, 4] and not f[2, 2:4].any()
    np.testing.assert_array_equal(oracle.forced_mask(5, 65, q_block=64), oracle.forced_mask(5, 65))


@pytest.mark.parametrize("S", [640, 679])
def test_qblock128_with_equal_halves_is_the_union_of_the_square_rows(S):
    # When the two 64-token halves of every query block hold the same tokens
    # (the second half reversed), the 128-token mean equals both 64-token
    # means exactly, so each 128-block row must be the union of the two square
    # rows (same thresholded set; diagonal {2i} or {2i+1}). A ragged 64-block
    # alone in the last query block keeps its square row.
    H, D = 2, 16
    rng = np.random.default_rng(5)
    qn = rng.standard_normal((1, S, H, D)).astype(np.float32)
    for b0 in range(0, S - 127, 128):
        qn[0, b0 + 64:b0 + 128] = qn[0, b0:b0 + 64][::-1]
    q = bf16(qn)
    k = bf16(rng.standard_normal((1, S, H, D)))
    for P, tau in ((0, 1.0), (100, 0.8), (0, 1.6)):
        sq = oracle.route_ref(q, k, P, tau)
        r = oracle.route_ref(q, k, P, tau, q_block=128)
        Nb = oracle.num_blocks(S)
        for i in range(Nb):
            pair = [j for j in (i - i % 2, i - i % 2 + 1) if j < Nb]
            union = np.logical_or.reduce([sq["kept"][:, :, j] for j in pair])
            np.testing.assert_array_equal(r["kept"][:, :, i], union)
            np.testing.assert_array_equal(r["p"][:, :, i], sq["p"][:, :, pair[0]])
        if S % 128:
            np.testing.assert_array_equal(r["kept"][:, :, Nb - 1], sq["kept"][:, :, Nb - 1])


def test_qblock128_route_invariants_and_modes():
    S, P = 1000, 130
    q, k, _ = sa_inputs.random_small(S, 2, 64, seed=3)
    Nb = oracle.num_blocks(S)
    r1 = oracle.route_ref(q, k, P, 1.0, q_block=128)
    r2 = oracle.route_ref(q, k, P, 2.0, q_block=128)
    assert r1["kept_q"].shape == (1, 2, 8, Nb) and r1["kept"].shape == (1, 2, Nb, Nb)
    for r in (r1, r2):
        kept = r["kept"]
        np.testing.assert_array_equal(kept[:, :, 0::2][:, :, :Nb // 2], kept[:, :, 1::2])
        assert kept[..., :3].all()                                 # sink columns
        for i in range(Nb):                                        # both key blocks of the diagonal
            assert kept[:, :, i, i - i % 2:min(Nb, i - i % 2 + 2)].all()
        assert not (r["ties"] & r["forced"]).any()
    assert not (r2["kept"] & ~r1["kept"]).any()                  # monotone in tau
    assert oracle.route_ref(q, k, P, 0.0, q_block=128)["kept"].all()
    dpq = oracle.route_ref(q, k, P, 1.0, q_block=128, mode="dense_prefix_queries")
    assert dpq["kept"][:, :, :4].all()                           # P = 130 meets query blocks 0, 1
    np.testing.assert_array_equal(dpq["kept"][:, :, 4:], r1["kept"][:, :, 4:])
    top = oracle.route_ref(q, k, P, 0.5, q_block=128, mode="top_mass")
    assert ((top["p"] * top["kept"]).sum(-1) >= 0.5 - 1e-12).all()
    with pytest.raises(ValueError):
        oracle.route_ref(q, k, P, 1.0, q_block=96)


# ------------------------------------------------ QK-norm + RoPE prologue --
# The fused prologue before attention ("Making MiniMax-H3 up to 9x faster on
# H100s", section "Custom kernels": QK-norm plus RoPE); the formulas are the
# oracle's reading (RMS norm over D with a weight vector, then rotation of
# interleaved pairs by tabulated angles).

def test_prologue_hand_example():
    x = np.zeros((1, 2, 1, 4))
    x[0, 0, 0] = [3.0, 4.0, 0.0, 0.0]        # mean square 6.25 -> 1/rms = 0.4
    x[0, 1, 0] = [0.0, 0.0, -1.0, 1.0]       # mean square 0.5
    gamma = np.array([1.0, 2.0, 3.0, 4.0])
    cos = np.array([[0.0, 1.0], [1.0, 0.0]])  # token 0: pair 0 turns by 90 degrees
    sin = np.array([[1.0, 0.0], [0.0, -1.0]]) # token 1: pair 1 turns by -90 degrees
    out = oracle.qk_prologue_ref(x, gamma, 0.0, cos, sin)
    # token 0: y = (1.2, 3.2, 0, 0); pair 0 (a, b) -> (-b, a)
    np.testing.assert_allclose(out[0, 0, 0], [-3.2, 1.2, 0.0, 0.0], rtol=0, atol=1e-12)
    # token 1: y = sqrt(2) * (0, 0, -3, 4); pair 1 (a, b) -> (b, -a)
    r2 = math.sqrt(2.0)
    np.testing.assert_allclose(out[0, 1, 0], [0.0, 0.0, 4 * r2, 3 * r2], rtol=0, atol=1e-12)


def test_prologue_norm_closed_forms():
    D, eps = 8, 1e-6
    x = np.full((1, 3, 2, D), -0.75)
    out = oracle.qk_prologue_ref(x, None, eps, None, None)
    np.testing.assert_allclose(out, -0.75 / math.sqrt(0.5625 + eps), rtol=1e-14)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((1, 5, 3, 16))
    out = oracle.qk_prologue_ref(x, None, eps, None, None)
    ms = (x * x).mean(-1)
    np.testing.assert_allclose((out * out).mean(-1), ms / (ms + eps), rtol=1e-12)
    g = rng.standard_normal(16)
    np.testing.assert_allclose(oracle.qk_prologue_ref(x, 2 * g, eps, None, None),
                               2 * oracle.qk_prologue_ref(x, g, eps, None, None), rtol=1e-14)


def test_prologue_rotation_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    S, H, D = 7, 2, 8
    x = rng.standard_normal((1, S, H, D))
    ang = rng.uniform(-4, 4, (S, D // 2))
    cos, sin = np.cos(ang), np.sin(ang)
    out = oracle.qk_prologue_ref(x, None, 1e-6, cos, sin)
    y = oracle.qk_prologue_ref(x, None, 1e-6, None, None)
    z = (y[..., 0::2] + 1j * y[..., 1::2]) * np.exp(1j * ang)[None, :, None, :]
    np.testing.assert_allclose(out[..., 0::2], z.real, atol=1e-12)
    np.testing.assert_allclose(out[..., 1::2], z.imag, atol=1e-12)
    ident = oracle.qk_prologue_ref(x, None, 1e-6, np.ones((S, D // 2)), np.zeros((S, D // 2)))
    np.testing.assert_array_equal(ident, y)
    # a rotation keeps each pair's length
    np.testing.assert_allclose(np.abs(z), np.hypot(y[..., 0::2], y[..., 1::2]), rtol=1e-12)


def test_prologue_rope_scores_depend_on_relative_position():
    # with the 1-D table theta = t * w, q_t . k_u depends on t - u only
    cfg = sa_inputs.get_config("tiny")
    cos, sin = (t.double().numpy() for t in sa_inputs.rope_tables(cfg))
    rng = np.random.default_rng(2)
    a, b = rng.standard_normal(cfg.D), rng.standard_normal(cfg.D)
    S = cfg.S

    def score(t, u):
        q = np.zeros((1, S, 1, cfg.D))
        k = np.zeros((1, S, 1, cfg.D))
        q[0, t, 0], k[0, u, 0] = a, b
        qo = oracle.qk_prologue_ref(q, None, 1e-6, cos, sin)[0, t, 0]
        ko = oracle.qk_prologue_ref(k, None, 1e-6, cos, sin)[0, u, 0]
        return float(qo @ ko)

    # tables are fp32, so equal up to their rounding
    assert abs(score(10, 3) - score(200, 193)) < 1e-4 * abs(score(10, 3)) + 1e-4
    assert abs(score(10, 3) - score(10, 40)) > 1e-3


# ----------------------------------------------- 8-bit scores (FP8 e4m3) --

def test_e4m3_decode_hand_values():
    # bytes worked out from the format: sign, 4 exponent bits (bias 7), 3 mantissa bits
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in cases.items():
        assert oracle.e4m3_decode(code) == val, hex(code)
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_round_hand_values():
    # ties go to the even mantissa; subnormals are spaced 2^-9
    x = [1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, 440.0, 447.0, 0.3, -1.0625, 1.9375]
    want = [1.0, 1.25, 2.0 ** -8, 0.0, 448.0, 448.0, 0.3125, -1.0, 2.0]
    assert oracle.e4m3_round(x).tolist() == want


def test_e4m3_round_is_the_nearest_value_by_brute_force():
    # against a search over every finite e4m3 value; ties take the even code
    codes = [c for c in range(256) if not math.isnan(oracle.e4m3_decode(c))]
    vals = np.array([oracle.e4m3_decode(c) for c in codes])
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1, 3000),
                        rng.normal(0, 2.0 ** -7, 2000), vals, (vals[:-1] + vals[1:]) / 2])
    x = x[np.abs(x) <= 448]
    got = oracle.e4m3_round(x)
    for xi, gi in zip(x, got):
        d = np.abs(vals - xi)
        near = vals[d == d.min()]
        if len(set(near.tolist()) - {0.0, -0.0}) > 1 or (len(near) > 1 and 0.0 not in near):
            # a tie: the value whose code has an even mantissa
            even = [v for v in near if (int(oracle.e4m3_encode([v])[0]) & 1) == 0]
            assert gi == even[0], (xi, gi, near)
        else:
            assert abs(gi) == abs(near[0]), (xi, gi, near)


def test_e4m3_round_agrees_with_torch_float8():
    # torch's own float8_e4m3fn conversion (round to nearest even) as a second opinion
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round(x.astype(np.float64)), t)


def test_e4m3_encode_inverts_decode():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v) or c == 0x80:
            continue
        assert int(oracle.e4m3_encode([v])[0]) == c


def test_fp8_block_exponent():
    assert [oracle.fp8_block_exponent(a) for a in (448.0, 449.0, 1.0, 1.75, 1.76, 0.0)] == \
        [0, 1, -8, -8, -7, 0]
    rng = np.random.default_rng(7)
    for a in np.exp(rng.uniform(-30, 30, 2000)):
        e = oracle.fp8_block_exponent(a)
        assert a / 2.0 ** e <= 448.0 < a / 2.0 ** (e - 1)      # the smallest such e


def test_quantize_blocks_are_independent_and_exact_on_the_grid():
    # block 0 holds e4m3 values (exponent 0 when its amax is 448), block 1 the
    # same values times 2^-5: both quantise to themselves, and the scales differ
    rng = np.random.default_rng(8)
    grid = np.array([oracle.e4m3_decode(c) for c in range(0x00, 0x7F)])
    a = rng.choice(grid, size=(64, 2, 16))
    a[0, 0, 0] = 448.0
    a[0, 1, 0] = 448.0
    x = np.concatenate([a, a * 2.0 ** -5], axis=0)[None]           # [1, 128, 2, 16]
    codes, exps, deq = oracle.quantize_qk_ref(x)
    assert exps[0, :, 0].tolist() == [0, 0] and exps[0, :, 1].tolist() == [-5, -5]
    assert np.array_equal(deq, x)
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    scale = np.repeat(2.0 ** exps[0].T, 64, axis=0)[None, :, :, None]   # [1, 128, 2, 1]
    assert np.array_equal(table[codes] * scale, x)


def test_fp8_attention_reduces_to_exact_attention_on_the_grid():
    # inputs already on each block's e4m3 grid: quantisation is the identity
    rng = np.random.default_rng(9)
    grid = np.array([oracle.e4m3_decode(c) for c in range(0x00, 0x7F)]) / 64.0
    S, H, D = 150, 2, 16
    q = rng.choice(grid, size=(1, S, H, D)) * rng.choice([-1, 1], size=(1, S, H, D))
    k = rng.choice(grid, size=(1, S, H, D)) * rng.choice([-1, 1], size=(1, S, H, D))
    v = rng.normal(size=(1, S, H, D))
    for x in (q, k):     # pin every block's amax to 448 / 64 so its exponent is -6
        for j in range(3):
            x[0, 64 * j, :, 0] = 7.0
    rp, ci = oracle.dense_csr(1, H, S)
    o8, l8 = oracle.attn_fp8_ref(q, k, v, rp, ci)
    o, l = oracle.attn_ref(q, k, v, rp, ci)
    assert np.allclose(o8, o, rtol=0, atol=1e-12) and np.allclose(l8, l, rtol=0, atol=1e-12)


def test_fp8_attention_sampled_items_equal_full():
    cfg, q, k, v = sa_inputs.make_inputs("tiny")
    ref = oracle.route_ref(q, k, cfg.P, float(np.float32(cfg.tau)))
    rp, ci = ref["row_ptr"], ref["col_idx"]
    o, l = oracle.attn_fp8_ref(q, k, v, rp, ci)
    items = [(0, 1, 0), (0, 3, 7), (0, 3, 15)]
    got = oracle.attn_fp8_ref(q, k, v, rp, ci, items=items)
    for (b, h, i), (oi, li) in got.items():
        assert np.array_equal(oi, o[b, 64 * i:64 * i + 64, h, :])
        assert np.array_equal(li, l[b, h, 64 * i:64 * i + 64])
    # and the 8-bit scores stay close to exact attention (a property, not a bound)
    oe, _ = oracle.attn_ref(q, k, v, rp, ci)
    assert np.linalg.norm(o - oe) / np.linalg.norm(oe) < 0.05
