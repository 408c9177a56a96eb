"""The C ABI on the host, without a GPU: the library builds and loads, exports
every function include/sa.h declares, sizes its buffers, and rejects bad
arguments before it would touch a device."""

import ctypes
import os
import re

import pytest

from helpers import lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sa():
    return lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z_]+)\s*\(", text)))


def test_header_declarations_are_all_exported(sa):
    names = declared_functions()
    assert len(names) >= 12
    L = sa.load_library()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(sa.EXPORTS) == names


def params(sa, B=1, S=38247, H=56, D=128, P=951, tau=1.0):
    p = sa.sa_params()
    sa.load_library().sa_params_init(ctypes.byref(p), B, S, H, D, P, tau)
    return p


def test_sizes(sa):
    L = sa.load_library()
    p = params(sa)
    assert L.sa_num_blocks(ctypes.byref(p)) == 598
    assert L.sa_route_rows(ctypes.byref(p)) == 56 * 598
    assert L.sa_route_max_nnz(ctypes.byref(p)) == 56 * 598 * 598
    a256 = lambda x: (x + 255) // 256 * 256
    vt = 56 * 128 * 38248 * 2                   # V repacked to fp16, key-contiguous
    cand = 56 * 598 * 64 * 2                    # pairing: 64 candidates per block (int16)
    tiles = 56 * 299 * 4                        # tile list
    assert L.sa_attn_workspace_bytes(ctypes.byref(p)) == a256(vt) + 256 + a256(cand) + a256(tiles)
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > 56 * 598 * 598 * 4
    p1 = params(sa, S=1, H=1, D=64, P=0)
    assert L.sa_num_blocks(ctypes.byref(p1)) == 1


@pytest.mark.parametrize("field,value,code", [
    ("D", 96, 2), ("D", 0, 1), ("block", 32, 1), ("S", 0, 1), ("prefix_len", -1, 1),
    ("prefix_len", 40000, 1), ("tau", -1.0, 1), ("tau", float("inf"), 1), ("H", 0, 1),
    ("softmax_scale", float("nan"), 1), ("route_mode", 3, 1), ("route_mode", -1, 1),
    ("q_block", 1, 1), ("q_block", 96, 1), ("q_block", 256, 1),
])
def test_bad_params_rejected_before_launch(sa, field, value, code):
    L = sa.load_library()
    p = params(sa)
    setattr(p, field, value)
    dummy = ctypes.c_void_p(256)
    assert L.sa_route(ctypes.byref(p), dummy, dummy, dummy, dummy, 10, dummy, 1 << 40,
                      None, None) == code
    assert L.sa_attn_dense(ctypes.byref(p), dummy, dummy, dummy, dummy, None, dummy, 1 << 40,
                           None, None) == code
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) == 0


def test_route_modes_and_their_tau_ranges(sa):
    L = sa.load_library()
    p = params(sa)
    assert p.route_mode == sa.SA_ROUTE_THRESHOLD           # what sa_params_init sets
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > 0
    p.route_mode = sa.SA_ROUTE_TOP_MASS
    p.tau = 1.0                                            # a mass: at most 1
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > 0
    p.tau = 1.5
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) == 0
    dummy = ctypes.c_void_p(256)
    assert L.sa_route(ctypes.byref(p), dummy, dummy, dummy, dummy, 10, dummy, 1 << 40,
                      None, None) == 1
    p.route_mode = sa.SA_ROUTE_DENSE_PREFIX_QUERIES         # a multiple of 1/Nb: any tau >= 0
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) > 0


def test_query_block_sizes_and_route_workspace(sa):
    L = sa.load_library()
    p = params(sa)
    assert p.q_block == 0                                  # what sa_params_init sets: 64
    square = L.sa_route_workspace_bytes(ctypes.byref(p))
    p.q_block = 64
    assert L.sa_route_workspace_bytes(ctypes.byref(p)) == square
    p.q_block = 128                                        # half the routed rows
    ws128 = L.sa_route_workspace_bytes(ctypes.byref(p))
    assert 0 < ws128 < square
    # the CSR is still one row per 64-token block, and attention needs the same workspace
    assert L.sa_route_rows(ctypes.byref(p)) == 56 * 598
    assert L.sa_route_max_nnz(ctypes.byref(p)) == 56 * 598 * 598
    p64 = params(sa)
    assert L.sa_attn_workspace_bytes(ctypes.byref(p)) == L.sa_attn_workspace_bytes(ctypes.byref(p64))


def test_null_and_misaligned_pointers_rejected(sa):
    L = sa.load_library()
    p = params(sa)
    a = ctypes.c_void_p(4096)
    assert L.sa_route(ctypes.byref(p), None, a, a, a, 10, a, 1 << 40, None, None) == 1
    # a missing pointer is reported before a short workspace
    assert L.sa_route(ctypes.byref(p), None, a, a, a, 10, a, 16, None, None) == 1
    assert L.sa_route(ctypes.byref(p), a, a, a, a, 10, a, 16, None, None) == 3
    assert L.sa_route(ctypes.byref(p), ctypes.c_void_p(4098), a, a, a, 10, a, 1 << 40,
                      None, None) == 1
    assert L.sa_route(ctypes.byref(p), a, a, a, a, 10, ctypes.c_void_p(4096 + 16), 1 << 40,
                      None, None) == 1  # workspace must be 256-byte aligned
    assert L.sa_attn_sparse(ctypes.byref(p), a, a, a, None, a, a, None, a, 1 << 40,
                            None, None) == 1
    assert L.sa_route(None, a, a, a, a, 10, a, 1 << 40, None, None) == 1


def test_small_workspace_and_bad_strides(sa):
    L = sa.load_library()
    p = params(sa)
    a = ctypes.c_void_p(4096)
    need = L.sa_route_workspace_bytes(ctypes.byref(p))
    assert L.sa_route(ctypes.byref(p), a, a, a, a, 10, a, need - 1, None, None) == 3
    need = L.sa_attn_workspace_bytes(ctypes.byref(p))
    assert L.sa_attn_dense(ctypes.byref(p), a, a, a, a, None, a, need - 1, None, None) == 3
    p.k_stride[1] = 7168 + 4   # not a multiple of 8 elements
    assert L.sa_route(ctypes.byref(p), a, a, a, a, 10, a, 1 << 40, None, None) == 1


def test_forward_host_requires_contiguous_layout(sa):
    L = sa.load_library()
    p = params(sa)
    p.q_stride[2] = 256
    a = ctypes.c_void_p(4096)
    args = [a] * 12
    assert L.sa_forward_host(ctypes.byref(p), *args, 10, a, 1 << 40, None, None) == 1


def test_status_strings_and_decode(sa):
    L = sa.load_library()
    assert L.sa_status_string(0) == b"SA_OK"
    assert L.sa_status_string(5) == b"SA_ERR_TIMEOUT"
    assert L.sa_dev_status_decode(0) == 0
    assert L.sa_dev_status_decode(sa.SA_DEV_TIMEOUT | sa.SA_DEV_CAPACITY) == 5
    assert L.sa_dev_status_decode(sa.SA_DEV_CAPACITY) == 3


def test_binding_refuses_cpu_tensors(sa):
    import torch
    q = torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sa.sa_route(q, q, 0, 1.0)
    with pytest.raises(ValueError):
        sa.sa_attn_dense(q, q, q)


def test_prologue_and_pooled_route_reject_bad_arguments(sa):
    L = sa.load_library()
    p = params(sa)
    a = ctypes.c_void_p(4096)
    f = ctypes.c_void_p(8192)
    big = 1 << 40

    def pro(**kw):
        args = dict(qi=a, ki=a, gq=None, gk=None, eps=1e-6, cs=None, sn=None, qo=a, ko=a,
                    ws=a, wsb=big)
        args.update(kw)
        return L.sa_qk_prologue(ctypes.byref(p), args["qi"], args["ki"], args["gq"], args["gk"],
                                args["eps"], args["cs"], args["sn"], args["qo"], args["ko"],
                                args["ws"], args["wsb"], None, None)

    assert pro(eps=-1.0) == 1
    assert pro(eps=float("nan")) == 1
    assert pro(cs=f) == 1                                # one table without the other
    assert pro(cs=f, sn=ctypes.c_void_p(8192 + 4)) == 1  # misaligned table
    assert pro(gq=ctypes.c_void_p(8192 + 8)) == 1        # misaligned weights
    assert pro(qo=None) == 1
    assert pro(ki=ctypes.c_void_p(4096 + 2)) == 1
    assert pro(ws=ctypes.c_void_p(4096 + 16)) == 1       # workspace not 256-byte aligned
    assert pro(wsb=1024) == 3                            # workspace too small
    assert L.sa_route_pooled(ctypes.byref(p), None, a, 10, a, big, None, None) == 1
    assert L.sa_route_pooled(ctypes.byref(p), a, a, 10, a, 1024, None, None) == 3
    p.D = 96
    assert pro() == 2
    assert L.sa_route_pooled(ctypes.byref(p), a, a, 10, a, big, None, None) == 2


def test_more_key_blocks_than_a_walk_holds_is_unsupported(sa):
    L = sa.load_library()
    p = params(sa, S=4096 * 64 + 1, H=1)          # 4097 key blocks
    a = ctypes.c_void_p(4096)
    assert L.sa_attn_dense(ctypes.byref(p), a, a, a, a, None, a, 1 << 40, None, None) == 2
    assert L.sa_attn_sparse(ctypes.byref(p), a, a, a, a, a, a, None, a, 1 << 40, None, None) == 2
    p = params(sa, S=4096 * 64, H=1)              # 4096: accepted up to the launch
    assert L.sa_attn_workspace_bytes(ctypes.byref(p)) > 0


def test_wait_check_needs_a_status_word(sa):
    L = sa.load_library()
    assert L.sa_check_wait_timeout(None, None) == 1


def test_prepare_and_run_check_their_own_arguments(sa):
    L = sa.load_library()
    p = params(sa)
    a = ctypes.c_void_p(4096)
    big = 1 << 40
    assert L.sa_attn_prepare(ctypes.byref(p), None, a, a, a, big, None, None) == 1   # no V
    assert L.sa_attn_prepare(ctypes.byref(p), a, None, a, a, big, None, None) == 1   # no route
    assert L.sa_attn_prepare(ctypes.byref(p), a, a, a, a, 1024, None, None) == 3     # short ws
    assert L.sa_attn_run(ctypes.byref(p), None, a, a, a, a, None, a, big, None, None) == 1
    assert L.sa_attn_run(ctypes.byref(p), a, a, a, a, None, None, a, big, None, None) == 1
    assert L.sa_attn_run(ctypes.byref(p), a, a, a, a, a, None, a, 1024, None, None) == 3


@pytest.mark.parametrize("S,q_block,max_heads", [(38247, 0, 9), (8192, 0, 72), (112640, 0, 1),
                                                 (38247, 128, 15), (8192, 128, 101),
                                                 (112640, 128, 3)])
def test_static_route_limits_stated_in_the_header(sa, S, q_block, max_heads):
    # the largest head counts sa.h states for sa_route_static's scratch array
    L = sa.load_library()

    def need(H):
        p = params(sa, S=S, H=H, P=0)
        p.q_block = q_block
        return L.sa_route_workspace_bytes(ctypes.byref(p))

    assert need(max_heads) <= sa.SA_ROUTE_STATIC_WS_BYTES < need(max_heads + 1)
