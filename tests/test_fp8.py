"""GPU parity of the 8-bit score path (sa_params.qk_format = SA_QK_FP8).

The reading (MiniAcc blog, "What is SageAttention?": 8-bit score
computation): Q and K quantised to e4m3 per (batch, head, 64-token block)
with a power-of-two scale, attention over the dequantised values. The
quantiser is integer/byte work and must match the oracle's bit for bit. The
attention is then compared with the oracle's quantise-then-attend result
under the same tolerances as the bf16 path: with the quantisation taken
exactly on both sides, what remains is the kernel's own fp32/fp16
arithmetic, which the 8-bit codes do not change (e4m3 x e4m3 products are
exact in fp32).
"""

import numpy as np
import pytest
import torch

import oracle
import sa_inputs
from helpers import (L2_TOL, MAXABS_TOL, f32, gather_rows, lib, lse_ok, out_errors, ref_rows,
                     sample_items, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return lib()


def new_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def quantize_gpu(sa, q, k):
    st = new_status()
    q8, k8, qe, ke = sa.sa_qk_quantize(q.cuda(), k.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return (q8.cpu().numpy(), k8.cpu().numpy(), qe.cpu().numpy().astype(np.int64),
            ke.cpu().numpy().astype(np.int64))


def check_codes(sa, q, k, heads=None):
    q8, k8, qe, ke = quantize_gpu(sa, q, k)
    for x, codes, exps in ((q, q8, qe), (k, k8, ke)):
        rc, re, _ = oracle.quantize_qk_ref(x, heads)
        hs = list(range(x.shape[2])) if heads is None else list(heads)
        assert np.array_equal(exps[:, hs, :], re)
        got = codes[:, :, hs, :]
        # -0 and +0 are the same value; compare codes with the sign of zero dropped
        got = np.where(got == 0x80, 0, got)
        assert np.array_equal(got, rc)


@pytest.mark.parametrize("S,H", [(64, 1), (200, 2), (1000, 3), (4096 + 17, 2)])
def test_quantized_codes_match_the_oracle_bit_for_bit(sa, S, H):
    q, k, _ = sa_inputs.random_small(S, H, 128, seed=S + H, std=3.0)
    check_codes(sa, q, k)


def test_quantized_codes_of_zero_and_extreme_blocks(sa):
    # an all-zero block (exponent 0), a block of huge values and one of tiny
    # values (the scale spans both ways), a block holding 448 exactly
    q, k, _ = sa_inputs.random_small(256, 1, 128, seed=5)
    q[:, 0:64] = 0
    q[:, 64:128] *= 2.0 ** 40
    q[:, 128:192] *= 2.0 ** -40
    k[:, 192:256] = 0
    k[0, 200, 0, 7] = 448.0
    check_codes(sa, q, k)


def gpu_route(sa, q, k, P, tau, q_block=64):
    st = new_status()
    rp, ci = sa.sa_route(q.cuda(), k.cuda(), P, tau, q_block=q_block, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rp = to_np(rp).astype(np.int64)
    return rp, to_np(ci).astype(np.int64)[: rp[-1]]


def gpu_attn_fp8(sa, q, k, v, rp=None, ci=None, q_block=64):
    st = new_status()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if rp is None:
        o, lse = sa.sa_attn_dense(qd, kd, vd, qk_format="fp8", dev_status=st)
    else:
        rpd = torch.as_tensor(rp, dtype=torch.int32, device="cuda")
        cid = torch.as_tensor(ci, dtype=torch.int32, device="cuda")
        o, lse = sa.sa_attn_sparse(qd, kd, vd, rpd, cid, q_block=q_block, qk_format="fp8",
                                   dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return to_np(o), to_np(lse)


@pytest.mark.parametrize("S,H,P,tau", [(50, 2, 50, 1.0), (65, 2, 0, 1.0), (200, 1, 0, 0.0),
                                       (1000, 3, 100, 1.0), (2048 + 33, 2, 64, 1.05)])
def test_fp8_attention_small_shapes(sa, S, H, P, tau):
    q, k, v = sa_inputs.random_small(S, H, 128, seed=S + 7)
    rp, ci = gpu_route(sa, q, k, P, tau)
    o, lse = gpu_attn_fp8(sa, q, k, v, rp, ci)
    o_ref, lse_ref = oracle.attn_fp8_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(lse, lse_ref)


def test_fp8_dense_small(sa):
    q, k, v = sa_inputs.random_small(700, 2, 128, seed=77)
    o, lse = gpu_attn_fp8(sa, q, k, v)
    rp, ci = oracle.dense_csr(1, 2, 700)
    o_ref, lse_ref = oracle.attn_fp8_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(lse, lse_ref)


@pytest.mark.parametrize("q_block", [64, 128])
def test_fp8_mid_full(sa, q_block):
    cfg, q, k, v = sa_inputs.make_inputs("mid")
    rp, ci = gpu_route(sa, q, k, cfg.P, cfg.tau, q_block=q_block)
    o, lse = gpu_attn_fp8(sa, q, k, v, rp, ci, q_block=q_block)
    o_ref, lse_ref = oracle.attn_fp8_ref(q, k, v, rp, ci)
    l2, mx, _ = out_errors(o, o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(lse, lse_ref)
    # the 8-bit scores themselves stay near exact attention (reported, loose)
    o_exact, _ = oracle.attn_ref(q, k, v, rp, ci)
    assert np.linalg.norm(o - o_exact) / np.linalg.norm(o_exact) < 0.05


def test_fp8_release_sampled(sa):
    cfg, q, k, v = sa_inputs.make_inputs("release")
    rp, ci = gpu_route(sa, q, k, cfg.P, cfg.tau)
    o, lse = gpu_attn_fp8(sa, q, k, v, rp, ci)
    Nb, n_sink = cfg.Nb, (cfg.P + 63) // 64
    items = sample_items(1, cfg.H, Nb, 4, 12, seed=11, must=(0, n_sink - 1, Nb - 1))
    check_codes(sa, q, k, heads=sorted({h for (_, h, _) in items}))
    ref = oracle.attn_fp8_ref(q, k, v, rp, ci, items=items)
    o_g, l_g = gather_rows(o, lse, items, cfg.S)
    o_r, l_r = ref_rows(ref, items)
    l2, mx, _ = out_errors(o_g, o_r)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(l_g, l_r)


def test_fp8_needs_head_dim_128(sa):
    q, k, v = sa_inputs.random_small(128, 1, 64, seed=3)
    with pytest.raises(sa.SaError):
        sa.sa_attn_dense(q.cuda(), k.cuda(), v.cuda(), qk_format="fp8")


def test_fp8_batch_and_strided_views(sa):
    # B = 2, heads 1..3 of a 5-head buffer: the quantiser reads strided Q and K
    # and the codes it writes are contiguous
    g = torch.Generator().manual_seed(18)
    big = [torch.randn((2, 300, 5, 128), generator=g).to(torch.bfloat16) for _ in range(3)]
    q, k, v = (t[:, :, 1:4, :] for t in big)
    qd, kd, vd = (t.cuda()[:, :, 1:4, :] for t in big)
    assert not qd.is_contiguous()
    st = new_status()
    rp, ci = sa.sa_route(qd, kd, 70, 1.0, dev_status=st)
    o = torch.empty((2, 300, 3, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, o=o, qk_format="fp8", dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rpn = to_np(rp).astype(np.int64)
    cin = to_np(ci).astype(np.int64)[: rpn[-1]]
    o_ref, lse_ref = oracle.attn_fp8_ref(q, k, v, rpn, cin)
    l2, mx, _ = out_errors(to_np(o), o_ref)
    assert l2 <= L2_TOL and mx <= MAXABS_TOL, (l2, mx)
    assert lse_ok(to_np(lse), lse_ref)
    check_codes(sa, q.contiguous(), k.contiguous())


@pytest.mark.parametrize("q_block", [64, 128])
def test_fp8_prepare_then_run_equals_attn_sparse(sa, q_block):
    # the two halves (the quantiser runs in sa_attn_run) give the one-call
    # result bit for bit
    cfg, q, k, v = sa_inputs.make_inputs("mid")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    st = new_status()
    rp, ci = sa.sa_route(qd, kd, cfg.P, cfg.tau, q_block=q_block, dev_status=st)
    o, lse = sa.sa_attn_sparse(qd, kd, vd, rp, ci, q_block=q_block, qk_format="fp8",
                               dev_status=st)
    p = sa.make_params(qd, kd, vd, o, q_block=q_block, qk_format="fp8")
    ws = torch.empty(sa.sa_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    sa.sa_attn_prepare(vd, rp, ci, workspace=ws, q_block=q_block, qk_format="fp8",
                       dev_status=st)
    o2, lse2 = sa.sa_attn_run(qd, kd, rp, ci, workspace=ws, v_like=vd, q_block=q_block,
                              qk_format="fp8", dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
