"""sa_route_static, the router for callers that cannot allocate device memory
(for example a plugin inside an inference engine that has reserved all of HBM
for its own pool): it runs on a scratch array the library owns instead of a
caller workspace. Checked through the C ABI against sa_route on the same
inputs, on calls made back to back, so the second call finds the first call's
leftovers in the shared array. This file is collected last on purpose."""

import ctypes

import pytest
import torch

import sa_inputs
from helpers import lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


def regular_route(sa, q, k, cfg, tau, mode, q_block):
    rp, ci = sa.sa_route(q, k, cfg.P, tau, mode=mode, q_block=q_block)
    torch.cuda.synchronize()
    return rp, ci


def static_route(sa, q, k, cfg, tau, mode, q_block, cap):
    L = sa.load_library()
    p = sa.make_params(q, k, prefix_len=cfg.P, tau=tau, mode=mode, q_block=q_block)
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) <= sa.SA_ROUTE_STATIC_WS_BYTES
    rows = int(L.sa_route_rows(ctypes.byref(p)))
    rp = torch.full((rows + 1,), -7, dtype=torch.int32, device="cuda")
    ci = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = L.sa_route_static(ctypes.byref(p), q.data_ptr(), k.data_ptr(), rp.data_ptr(),
                             ci.data_ptr(), cap, st.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert code == 0, sa._status_name(code)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return rp, ci


# Each sequence runs back to back on the one shared array, so every call
# after the first starts from what a call of another shape, reading or
# query block size left there.
SEQUENCES = {
    "threshold": [("mid", None, "threshold", 64), ("mid", None, "threshold", 64),
                  ("tiny", None, "threshold", 64)],
    "readings_and_query_blocks": [("mid", 0.85, "top_mass", 64), ("mid", None, "threshold", 128),
                                  ("tiny", None, "dense_prefix_queries", 64),
                                  ("mid", 0.85, "top_mass", 128), ("tiny", None, "threshold", 64)],
}


@pytest.mark.parametrize("seq", sorted(SEQUENCES))
def test_static_route_matches_sa_route_on_consecutive_calls(sa, seq):
    runs = []
    for name, tau, mode, q_block in SEQUENCES[seq]:
        cfg, q, k, _ = sa_inputs.make_inputs(name)
        runs.append((cfg, q.cuda(), k.cuda(), cfg.tau if tau is None else tau, mode, q_block))
    for cfg, q, k, tau, mode, q_block in runs:
        ref_rp, ref_ci = regular_route(sa, q, k, cfg, tau, mode, q_block)
        rp, ci = static_route(sa, q, k, cfg, tau, mode, q_block, ref_ci.numel())
        assert torch.equal(rp, ref_rp)
        n = int(ref_rp[-1].item())
        assert torch.equal(ci[:n], ref_ci[:n])


def test_static_route_rejects_shapes_beyond_its_scratch(sa):
    L = sa.load_library()
    p = sa.sa_params()
    L.sa_params_init(ctypes.byref(p), 1, 38247, 56, 128, 951, 1.0)  # needs ~180 MiB
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > sa.SA_ROUTE_STATIC_WS_BYTES
    buf = torch.empty(1024, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    code = L.sa_route_static(ctypes.byref(p), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                             buf.data_ptr(), 16, None, stream)
    assert code == 3  # SA_ERR_CAPACITY
    # a missing pointer is reported before the capacity, as sa_route does
    code = L.sa_route_static(ctypes.byref(p), buf.data_ptr(), None, buf.data_ptr(),
                             buf.data_ptr(), 16, None, stream)
    assert code == 1  # SA_ERR_INVALID_ARG
