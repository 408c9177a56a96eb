"""GPU parity of the router's other readings (sa_params.route_mode).

The pages leave the router rule open; besides the default threshold rule the
library offers dense prefix query rows and top-mass selection (sa.h,
SA_ROUTE_*). Each is checked like the default: the CUDA route equals the
oracle's kept sets outside the oracle's ties, and attention over the CUDA
route matches the oracle within the tolerances of ``helpers``.
"""

import numpy as np
import pytest
import torch

import oracle
import sa_inputs
from helpers import L2_TOL, MAXABS_TOL, compare_route, f32, lib, lse_ok, out_errors, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


def route_both(sa, q, k, P, tau, mode):
    B, S, H, D = q.shape
    Nb = oracle.num_blocks(S)
    ref = oracle.route_ref(q, k, P, f32(tau), mode=mode)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rp, ci = sa.sa_route(q.cuda(), k.cuda(), P, tau, mode=mode, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rp, ci = to_np(rp).astype(np.int64), to_np(ci).astype(np.int64)
    bad, ties = compare_route(rp, ci[:rp[-1]], ref, B, H, Nb)
    assert bad == 0, f"{bad} decisions differ outside ties ({ties} ties)"
    return ref, rp, ci[:rp[-1]]


def attn_check(sa, q, k, v, rp, ci):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rpd = torch.as_tensor(rp, dtype=torch.int32, device="cuda")
    cid = torch.as_tensor(ci, dtype=torch.int32, device="cuda")
    o, lse = sa.sa_attn_sparse(q.cuda(), k.cuda(), v.cuda(), rpd, cid, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, lse_ref = oracle.attn_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL and lse_ok(to_np(lse), lse_ref)


SMALL = [  # (S, H, D, P, tau)
    (1, 2, 64, 0, 0.5),
    (65, 2, 128, 0, 0.5),
    (383, 2, 128, 100, 0.7),
    (640, 2, 64, 0, 0.0),
    (640, 2, 64, 64, 1.0),
    (1000, 2, 128, 951, 0.3),
    (2047, 1, 64, 200, 0.9),
]


@pytest.mark.parametrize("S,H,D,P,tau", SMALL)
def test_top_mass_small_shapes(sa, S, H, D, P, tau):
    q, k, v = sa_inputs.random_small(S, H, D, seed=S + 7 * H + D)
    _, rp, ci = route_both(sa, q, k, P, tau, "top_mass")
    attn_check(sa, q, k, v, rp, ci)


@pytest.mark.parametrize("S,H,D,P", [(1, 1, 64, 0), (383, 2, 128, 100), (1000, 2, 64, 951),
                                     (2047, 1, 128, 130)])
def test_dense_prefix_queries_small_shapes(sa, S, H, D, P):
    q, k, v = sa_inputs.random_small(S, H, D, seed=S + 11 * H)
    ref, rp, ci = route_both(sa, q, k, P, 1.0, "dense_prefix_queries")
    n_sink = (P + 63) // 64
    assert ref["kept"][:, :, :n_sink, :].all()
    attn_check(sa, q, k, v, rp, ci)


@pytest.mark.parametrize("mode,tau", [("top_mass", 0.3), ("top_mass", 0.7), ("top_mass", 0.9),
                                      ("dense_prefix_queries", None)])
def test_tiny_and_mid_modes(sa, mode, tau):
    for name in ("tiny", "mid"):
        cfg, q, k, v = sa_inputs.make_inputs(name)
        t = cfg.tau if tau is None else tau
        _, rp, ci = route_both(sa, q, k, cfg.P, t, mode)
        if name == "tiny":
            attn_check(sa, q, k, v, rp, ci)


def test_top_mass_release_route_bitexact(sa):
    cfg, q, k, _ = sa_inputs.make_inputs("release")
    ref, _, _ = route_both(sa, q, k, cfg.P, 0.75, "top_mass")
    d = oracle.block_density(ref["kept"])
    assert 0.05 < d < 0.6, d
