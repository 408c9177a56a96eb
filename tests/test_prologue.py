"""GPU parity of the fused QK-norm + RoPE prologue (sa_qk_prologue) and the
route from its pooled block means (sa_route_pooled).

The outputs are the exact (fp64) QK-norm + RoPE of the oracle rounded to bf16
by the kernel from an fp32 computation. Each element must lie within one bf16
ulp of the exact value plus the fp32 forward error of its rotation, which
scales with the magnitude of the rotated terms, 2e-6 (|y_a c| + |y_b s|):
the normalised y carry a relative error of about 7e-7 (sum of squares, the
reciprocal square root to 2 ulp, two products) and the rotation adds a few
fp32 roundings; where the two products nearly cancel, the result is far
smaller than its terms. All but a small fraction must be the nearest bf16.

The pooled means the prologue leaves behind must route exactly as sa_route
does from the prologue's own outputs (the same bf16 values summed the same
way), and as the oracle does on them outside its ties.
"""

import numpy as np
import pytest
import torch

import oracle
import sa_inputs
from helpers import compare_route, f32, lib, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    return np.exp2(np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)


def check_faithful(gpu: np.ndarray, exact: np.ndarray, mag: np.ndarray,
                   frac_tol: float = 1e-3):
    """Every element within one bf16 ulp of the exact value plus the fp32
    forward error 2e-6 * mag; at most a small fraction further than half an
    ulp plus that error (not the nearest bf16)."""
    err = np.abs(gpu - exact)
    ulp = bf16_ulp(exact)
    fp32 = 2e-6 * mag
    tiny = (np.abs(exact) < 1e-30) & (mag < 1e-30)
    assert np.all(np.where(tiny, np.abs(gpu) <= 1e-30, err <= ulp * (1 + 1e-9) + fp32)), \
        float(np.max(np.where(tiny, 0, err / (ulp + fp32))))
    off = int(np.sum(~tiny & (err > 0.5 * ulp * (1 + 1e-6) + fp32)))
    assert off <= max(2, frac_tol * exact.size), (off, exact.size)


def inputs(S, H, D, seed, with_gamma=True, with_rope=True):
    q, k, v = sa_inputs.random_small(S, H, D, seed=seed)
    gq, gk = sa_inputs.qk_norm_weights(D, seed=seed) if with_gamma else (None, None)
    if with_rope:
        cfg = sa_inputs.Config("t", S=S, P=0, H=H, D=D, tau=1.0, kind="iid")
        cos, sin = sa_inputs.rope_tables(cfg)
    else:
        cos = sin = None
    return q, k, v, gq, gk, cos, sin


def run_prologue(sa, q, k, gq, gk, eps, cos, sin, q_block=64, in_place=False):
    dev = lambda t: None if t is None else t.cuda()
    qd, kd = q.cuda(), k.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {"q_out": qd, "k_out": kd} if in_place else {}
    qo, ko, ws = sa.sa_qk_prologue(qd, kd, dev(gq), dev(gk), eps, dev(cos), dev(sin),
                                   q_block=q_block, dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return qo, ko, ws


def np_or_none(t):
    return None if t is None else t.double().numpy()


def check_outputs(q, k, qo, ko, gq, gk, eps, cos, sin):
    c, s = np_or_none(cos), np_or_none(sin)
    for x, out, g in ((q, qo, gq), (k, ko, gk)):
        exact = oracle.qk_prologue_ref(x, np_or_none(g), eps, c, s)
        y = np.abs(oracle.qk_prologue_ref(x, np_or_none(g), eps, None, None))
        if c is None:
            mag = y
        else:                               # |y_a c| + |y_b s| of each output of a pair
            ac, as_ = np.abs(c)[None, :, None, :], np.abs(s)[None, :, None, :]
            mag = np.empty_like(y)
            mag[..., 0::2] = y[..., 0::2] * ac + y[..., 1::2] * as_
            mag[..., 1::2] = y[..., 0::2] * as_ + y[..., 1::2] * ac
        check_faithful(to_np(out), exact, mag)


def check_routes(sa, qo, ko, ws, P, tau, q_block, mode="threshold"):
    B, S, H, _ = qo.shape
    Nb = oracle.num_blocks(S)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rp1, ci1 = sa.sa_route_pooled(qo, ws, P, tau, k=ko, mode=mode, q_block=q_block, dev_status=st)
    rp2, ci2 = sa.sa_route(qo, ko, P, tau, mode=mode, q_block=q_block, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rp1, rp2 = to_np(rp1).astype(np.int64), to_np(rp2).astype(np.int64)
    assert np.array_equal(rp1, rp2)
    ci1, ci2 = to_np(ci1)[:rp1[-1]].astype(np.int64), to_np(ci2)[:rp2[-1]].astype(np.int64)
    assert np.array_equal(ci1, ci2)
    return rp1, ci1, Nb


SMALL = [  # (S, H, D, q_block, gamma, rope, P, tau)
    (1, 1, 64, 64, True, True, 0, 1.0),
    (65, 2, 128, 64, True, False, 0, 0.7),
    (127, 1, 64, 128, False, True, 64, 1.0),
    (383, 3, 64, 64, True, True, 100, 1.0),
    (1000, 2, 128, 128, True, True, 951, 0.5),
    (2047, 1, 128, 64, False, False, 200, 1.3),
]


@pytest.mark.parametrize("S,H,D,qb,g,r,P,tau", SMALL)
def test_small_shapes_outputs_and_route(sa, S, H, D, qb, g, r, P, tau):
    q, k, _, gq, gk, cos, sin = inputs(S, H, D, seed=S + H + D, with_gamma=g, with_rope=r)
    eps = 1e-6
    qo, ko, ws = run_prologue(sa, q, k, gq, gk, eps, cos, sin, q_block=qb)
    check_outputs(q, k, qo, ko, gq, gk, eps, cos, sin)
    rp, ci, Nb = check_routes(sa, qo, ko, ws, P, tau, qb)
    ref = oracle.route_ref(qo.cpu(), ko.cpu(), P, f32(tau), q_block=qb)
    bad, ties = compare_route(rp, ci, ref, 1, H, Nb)
    assert bad == 0, (bad, ties)


def test_in_place_equals_out_of_place(sa):
    q, k, _, gq, gk, cos, sin = inputs(700, 2, 128, seed=3)
    qo, ko, _ = run_prologue(sa, q, k, gq, gk, 1e-6, cos, sin)
    qi, ki, _ = run_prologue(sa, q, k, gq, gk, 1e-6, cos, sin, in_place=True)
    assert torch.equal(qo.view(torch.int16), qi.view(torch.int16))
    assert torch.equal(ko.view(torch.int16), ki.view(torch.int16))


def test_zero_vectors_and_other_modes(sa):
    q, k, _, gq, gk, cos, sin = inputs(500, 2, 64, seed=9)
    q[:, 100:300] = 0                       # whole blocks of zero vectors: output 0
    qo, ko, ws = run_prologue(sa, q, k, gq, gk, 1e-5, cos, sin)
    assert not torch.any(qo[:, 100:300].float() != 0)
    check_outputs(q, k, qo, ko, gq, gk, 1e-5, cos, sin)
    for mode, tau in (("dense_prefix_queries", 1.0), ("top_mass", 0.6)):
        check_routes(sa, qo, ko, ws, 130, tau, 64, mode=mode)


@pytest.mark.parametrize("qb", [64, 128])
def test_release_prologue_route_and_sampled_outputs(sa, qb):
    cfg, q, k, _ = sa_inputs.make_inputs("release")
    gq, gk = sa_inputs.qk_norm_weights(cfg.D)
    cos, sin = sa_inputs.rope_tables(cfg)
    qo, ko, ws = run_prologue(sa, q, k, gq, gk, 1e-6, cos, sin, q_block=qb)
    rp, ci, Nb = check_routes(sa, qo, ko, ws, cfg.P, cfg.tau, qb)
    d = float(rp[-1]) / (cfg.H * Nb * Nb)
    assert 0.0 < d <= 1.0
    heads = [0, 31, 55]
    sub = lambda t: t[:, :, heads].contiguous()
    check_outputs(sub(q), sub(k), sub(qo.cpu()), sub(ko.cpu()), gq, gk, 1e-6, cos, sin)


def test_batch_and_strided_views(sa):
    # B = 2, heads 1..3 of a 5-head buffer: non-contiguous b/s/h strides, out of place
    # into tensors of the same strides, and in place
    S, D = 300, 128
    g = torch.Generator().manual_seed(21)
    big = [torch.randn((2, S, 5, D), generator=g).to(torch.bfloat16) for _ in range(2)]
    q, k = (t[:, :, 1:4, :] for t in big)
    gq, gk = sa_inputs.qk_norm_weights(D, seed=4)
    cfg = sa_inputs.Config("t", S=S, P=0, H=3, D=D, tau=1.0, kind="iid")
    cos, sin = sa_inputs.rope_tables(cfg)
    bigd = [t.cuda() for t in big]
    qd, kd = (t[:, :, 1:4, :] for t in bigd)
    assert not qd.is_contiguous()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo, ko, ws = sa.sa_qk_prologue(qd, kd, gq.cuda(), gk.cuda(), 1e-6, cos.cuda(), sin.cuda(),
                                   dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and qo.stride() == qd.stride()
    check_outputs(q, k, qo, ko, gq, gk, 1e-6, cos, sin)
    check_routes(sa, qo, ko, ws, 64, 1.0, 64)
    sa.sa_qk_prologue(qd, kd, gq.cuda(), gk.cuda(), 1e-6, cos.cuda(), sin.cuda(), q_out=qd,
                      k_out=kd, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(qd.view(torch.int16), qo.view(torch.int16))
    assert torch.equal(kd.view(torch.int16), ko.view(torch.int16))
    # the other heads of the buffers are untouched
    for t, td in zip(big, bigd):
        for h in (0, 4):
            assert torch.equal(td[:, :, h].cpu().view(torch.int16), t[:, :, h].view(torch.int16))
