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


def regular_route(sa, q, k, cfg):
    rp, ci = sa.sa_route(q, k, cfg.P, cfg.tau)
    torch.cuda.synchronize()
    return rp, ci


def static_route(sa, q, k, cfg, cap):
    L = sa.load_library()
    p = sa.make_params(q, k, prefix_len=cfg.P, tau=cfg.tau)
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


def test_static_route_matches_sa_route_on_consecutive_calls(sa):
    runs = []
    for name in ("mid", "mid", "tiny"):
        cfg, q, k, _ = sa_inputs.make_inputs(name)
        runs.append((cfg, q.cuda(), k.cuda()))
    for cfg, q, k in runs:
        ref_rp, ref_ci = regular_route(sa, q, k, cfg)
        rp, ci = static_route(sa, q, k, cfg, ref_ci.numel())
        assert torch.equal(rp, ref_rp)
        n = int(ref_rp[-1].item())
        assert torch.equal(ci[:n], ref_ci[:n])


def test_static_route_rejects_shapes_beyond_its_scratch(sa):
    L = sa.load_library()
    p = sa.sa_params()
    L.sa_params_init(ctypes.byref(p), 1, 38247, 56, 128, 951, 1.0)  # needs ~180 MiB
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > sa.SA_ROUTE_STATIC_WS_BYTES
    buf = torch.empty(1024, dtype=torch.int32, device="cuda")
    code = L.sa_route_static(ctypes.byref(p), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                             buf.data_ptr(), 16, None, torch.cuda.current_stream().cuda_stream)
    assert code == 3  # SA_ERR_CAPACITY
