"""Routed block-sparse self-attention on GB300 (sm_103a): Python binding.

This module only marshals arguments to the C ABI of ``libsa_gb300.so``
(declared in ``include/sa.h``): it reads tensor pointers, strides and the
current CUDA stream, allocates outputs with torch when the caller passes
none, and calls the library. Every step of routing and attention runs in the
library's CUDA kernels. There is no CPU path: if the library is missing or a
tensor is not on a CUDA device, the call raises.

Entry points (same names as the C ABI):
    sa_route(q, k, prefix_len, tau, ...)              -> (row_ptr, col_idx)
    sa_attn_sparse(q, k, v, row_ptr, col_idx, ...)    -> (o, lse)
    sa_attn_dense(q, k, v, ...)                       -> (o, lse)
    sa_qk_prologue(q, k, ...)                         -> (q_out, k_out, workspace)
    sa_qk_quantize(q, k, ...)                         -> (q8, k8, q_exp, k_exp)
    sa_route_pooled(q_out, workspace, prefix_len, tau, ...) -> (row_ptr, col_idx)
    sa_forward_host(q_host, k_host, v_host, ...)      -> o_host (+ lse_host)
Tensors are [B, S, H, D] bf16 with a contiguous last dimension.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "SaError", "load_library", "library_path", "sa_params", "make_params", "sa_route",
    "sa_qk_prologue", "sa_route_pooled", "sa_attn_prepare", "sa_attn_run",
    "sa_attn_sparse", "sa_attn_dense", "sa_forward_host", "sa_route_workspace_bytes",
    "sa_attn_workspace_bytes", "sa_route_max_nnz", "check_dev_status", "EXPORTS",
    "sa_qk_quantize", "SA_QK_BF16", "SA_QK_FP8", "QK_FORMATS",
    "SA_DEV_CAPACITY", "SA_DEV_TIMEOUT", "SA_DEV_BAD_ROUTE", "SA_DEV_RANGE",
    "SA_ROUTE_THRESHOLD", "SA_ROUTE_DENSE_PREFIX_QUERIES", "SA_ROUTE_TOP_MASS", "ROUTE_MODES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CAPACITY, SA_ERR_CUDA, SA_ERR_TIMEOUT = range(6)
SA_DEV_CAPACITY, SA_DEV_TIMEOUT, SA_DEV_BAD_ROUTE, SA_DEV_RANGE = 1, 2, 4, 8
# readings of the router rule (sa_params.route_mode)
SA_ROUTE_THRESHOLD, SA_ROUTE_DENSE_PREFIX_QUERIES, SA_ROUTE_TOP_MASS = 0, 1, 2
ROUTE_MODES = {"threshold": SA_ROUTE_THRESHOLD,
               "dense_prefix_queries": SA_ROUTE_DENSE_PREFIX_QUERIES,
               "top_mass": SA_ROUTE_TOP_MASS}
# arithmetic of the score product (sa_params.qk_format)
SA_QK_BF16, SA_QK_FP8 = 0, 1
QK_FORMATS = {"bf16": SA_QK_BF16, "fp8": SA_QK_FP8}

# Every function include/sa.h declares.
EXPORTS = (
    "sa_params_init", "sa_num_blocks", "sa_route_rows", "sa_route_max_nnz",
    "sa_route_workspace_bytes", "sa_route", "sa_attn_workspace_bytes", "sa_attn_sparse",
    "sa_attn_dense", "sa_forward_host", "sa_dev_status_decode", "sa_status_string",
    "sa_route_static", "sa_qk_prologue", "sa_route_pooled", "sa_check_wait_timeout",
    "sa_attn_prepare", "sa_attn_run", "sa_qk_quantize",
)
SA_ROUTE_STATIC_WS_BYTES = 32 << 20


class SaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_status_name(code)}")


class sa_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("S", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("block", ctypes.c_int32), ("prefix_len", ctypes.c_int32),
        ("tau", ctypes.c_float), ("softmax_scale", ctypes.c_float),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("route_mode", ctypes.c_int32), ("q_block", ctypes.c_int32),
        ("qk_format", ctypes.c_int32),
    ]


def library_path() -> str:
    return os.path.join(_PKG, "libsa_gb300.so")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (once) and type the shared library. Raises if it is missing."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or library_path()
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with `python -m block_sparse_attention_sa_gb300.build`")
    lib = ctypes.CDLL(p)
    P = ctypes.POINTER(sa_params)
    vp, i32p, i64, sz = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64, ctypes.c_size_t
    sig = {
        "sa_params_init": (None, [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_float]),
        "sa_num_blocks": (ctypes.c_int32, [P]),
        "sa_route_rows": (i64, [P]),
        "sa_route_max_nnz": (i64, [P]),
        "sa_route_workspace_bytes": (sz, [P]),
        "sa_attn_workspace_bytes": (sz, [P]),
        "sa_route": (ctypes.c_int, [P, vp, vp, vp, vp, i64, vp, sz, vp, vp]),
        "sa_route_static": (ctypes.c_int, [P, vp, vp, vp, vp, i64, vp, vp]),
        "sa_qk_prologue": (ctypes.c_int, [P, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp,
                                          sz, vp, vp]),
        "sa_route_pooled": (ctypes.c_int, [P, vp, vp, i64, vp, sz, vp, vp]),
        "sa_attn_sparse": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
        "sa_attn_dense": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
        "sa_forward_host": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64,
                                           vp, sz, vp, vp]),
        "sa_dev_status_decode": (ctypes.c_int, [ctypes.c_int32]),
        "sa_check_wait_timeout": (ctypes.c_int, [vp, vp]),
        "sa_attn_prepare": (ctypes.c_int, [P, vp, vp, vp, vp, sz, vp, vp]),
        "sa_attn_run": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
        "sa_qk_quantize": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp]),
        "sa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _status_name(code: int) -> str:
    try:
        return load_library().sa_status_string(code).decode()
    except Exception:  # library not loadable: still report the number
        return f"status {code}"


def _check(code: int, what: str) -> None:
    if code != SA_OK:
        raise SaError(code, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bshd_strides(t: torch.Tensor, name: str):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be [B, S, H, D] with a contiguous last dimension")
    return (t.stride(0), t.stride(1), t.stride(2))


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device: there is no CPU path")


def make_params(q: torch.Tensor, k: Optional[torch.Tensor] = None, v: Optional[torch.Tensor] = None,
                o: Optional[torch.Tensor] = None, prefix_len: int = 0, tau: float = 1.0,
                scale: float = 0.0, mode="threshold", q_block: int = 64,
                qk_format="bf16") -> sa_params:
    B, S, H, D = q.shape
    p = sa_params()
    p.B, p.S, p.H, p.D, p.block, p.q_block = B, S, H, D, 64, int(q_block)
    p.qk_format = QK_FORMATS[qk_format] if isinstance(qk_format, str) else int(qk_format)
    p.prefix_len, p.tau, p.softmax_scale = int(prefix_len), float(tau), float(scale)
    p.route_mode = ROUTE_MODES[mode] if isinstance(mode, str) else int(mode)
    for field, t in (("q_stride", q), ("k_stride", k if k is not None else q),
                     ("v_stride", v if v is not None else q), ("o_stride", o if o is not None else q)):
        st = _bshd_strides(t, field[0])
        arr = getattr(p, field)
        for i in range(3):
            arr[i] = st[i]
    return p


def sa_route_workspace_bytes(p: sa_params) -> int:
    return int(load_library().sa_route_workspace_bytes(ctypes.byref(p)))


def sa_attn_workspace_bytes(p: sa_params) -> int:
    return int(load_library().sa_attn_workspace_bytes(ctypes.byref(p)))


def sa_route_max_nnz(p: sa_params) -> int:
    return int(load_library().sa_route_max_nnz(ctypes.byref(p)))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]) -> torch.Tensor:
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def sa_route(q: torch.Tensor, k: torch.Tensor, prefix_len: int, tau: float, scale: float = 0.0, *,
             mode="threshold", q_block: int = 64, row_ptr: Optional[torch.Tensor] = None,
             col_idx: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             dev_status: Optional[torch.Tensor] = None,
             stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block route of every (b, h, query block): int32 row_ptr [B*H*Nb+1] and
    col_idx (capacity B*H*Nb*Nb unless given; valid entries are
    col_idx[:row_ptr[-1]]). ``mode``: "threshold", "dense_prefix_queries" or
    "top_mass" (the SA_ROUTE_* readings of sa.h). ``q_block``: 64, or 128 for
    128-token query blocks (rows 2i and 2i + 1 then hold the same list)."""
    _require_cuda(q, k)
    lib = load_library()
    p = make_params(q, k, prefix_len=prefix_len, tau=tau, scale=scale, mode=mode,
                    q_block=q_block)
    rows = int(lib.sa_route_rows(ctypes.byref(p)))
    if rows == 0:
        _check(SA_ERR_INVALID_ARG, "sa_route")
    if row_ptr is None:
        row_ptr = torch.empty(rows + 1, dtype=torch.int32, device=q.device)
    if col_idx is None:
        col_idx = torch.empty(sa_route_max_nnz(p), dtype=torch.int32, device=q.device)
    ws = _workspace(sa_route_workspace_bytes(p), q.device, workspace)
    code = lib.sa_route(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(row_ptr), _ptr(col_idx),
                        col_idx.numel(), _ptr(ws), ws.numel() * ws.element_size(),
                        _ptr(dev_status), _stream(stream))
    _check(code, "sa_route")
    return row_ptr, col_idx


def sa_qk_prologue(q: torch.Tensor, k: torch.Tensor, gamma_q: Optional[torch.Tensor] = None,
                   gamma_k: Optional[torch.Tensor] = None, eps: float = 1e-6,
                   cos: Optional[torch.Tensor] = None, sin: Optional[torch.Tensor] = None, *,
                   q_block: int = 64, q_out: Optional[torch.Tensor] = None,
                   k_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   dev_status: Optional[torch.Tensor] = None, stream=None):
    """QK-norm + RoPE of q, k (bf16 [B,S,H,D]) with the router's pooling fused
    in: returns (q_out, k_out, workspace); pass the workspace to
    sa_route_pooled. gamma_* fp32 [D] or None; cos, sin fp32 [S, D/2] or None.
    q_out/k_out default to new tensors with q/k's strides; pass q_out=q for in place."""
    _require_cuda(q, k, gamma_q, gamma_k, cos, sin)
    lib = load_library()
    if q_out is None:
        q_out = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    if k_out is None:
        k_out = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    if q_out.stride() != q.stride() or k_out.stride() != k.stride():
        raise ValueError("q_out / k_out must have the strides of q / k")
    for t, name in ((gamma_q, "gamma_q"), (gamma_k, "gamma_k"), (cos, "cos"), (sin, "sin")):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous fp32 tensor")
    p = make_params(q, k, q_block=q_block)
    ws = _workspace(sa_route_workspace_bytes(p), q.device, workspace)
    code = lib.sa_qk_prologue(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(gamma_q), _ptr(gamma_k),
                              float(eps), _ptr(cos), _ptr(sin), _ptr(q_out), _ptr(k_out), _ptr(ws),
                              ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream))
    _check(code, "sa_qk_prologue")
    return q_out, k_out, ws


def sa_route_pooled(q: torch.Tensor, workspace: torch.Tensor, prefix_len: int, tau: float,
                    scale: float = 0.0, *, k: Optional[torch.Tensor] = None, mode="threshold",
                    q_block: int = 64, row_ptr: Optional[torch.Tensor] = None,
                    col_idx: Optional[torch.Tensor] = None,
                    dev_status: Optional[torch.Tensor] = None, stream=None):
    """The route from the block means sa_qk_prologue left in ``workspace``;
    q (and k, default q's layout) give the shape and strides of that call."""
    _require_cuda(q, workspace)
    lib = load_library()
    p = make_params(q, k if k is not None else q, prefix_len=prefix_len, tau=tau, scale=scale,
                    mode=mode, q_block=q_block)
    rows = int(lib.sa_route_rows(ctypes.byref(p)))
    if rows == 0:
        _check(SA_ERR_INVALID_ARG, "sa_route_pooled")
    if row_ptr is None:
        row_ptr = torch.empty(rows + 1, dtype=torch.int32, device=q.device)
    if col_idx is None:
        col_idx = torch.empty(sa_route_max_nnz(p), dtype=torch.int32, device=q.device)
    code = lib.sa_route_pooled(ctypes.byref(p), _ptr(row_ptr), _ptr(col_idx), col_idx.numel(),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(dev_status), _stream(stream))
    _check(code, "sa_route_pooled")
    return row_ptr, col_idx


def _attn_out(q, o, lse, want_lse):
    B, S, H, D = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    return o, lse


def sa_attn_sparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, row_ptr: torch.Tensor,
                   col_idx: torch.Tensor, scale: float = 0.0, *, o: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                   workspace: Optional[torch.Tensor] = None, q_block: int = 64,
                   qk_format="bf16", dev_status: Optional[torch.Tensor] = None, stream=None):
    """Attention over the routed key blocks: (o bf16 [B,S,H,D], lse fp32 [B,H,S] or None).
    ``q_block`` = 128 when the route came from sa_route(..., q_block=128): the
    kernel's tiles are then the 128-token query blocks, with no pairing step.
    ``qk_format`` = "fp8" for 8-bit scores (see sa_qk_quantize)."""
    _require_cuda(q, k, v, row_ptr, col_idx)
    lib = load_library()
    o, lse = _attn_out(q, o, lse, want_lse)
    p = make_params(q, k, v, o, scale=scale, q_block=q_block, qk_format=qk_format)
    ws = _workspace(sa_attn_workspace_bytes(p), q.device, workspace)
    code = lib.sa_attn_sparse(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(row_ptr),
                              _ptr(col_idx), _ptr(o), _ptr(lse), _ptr(ws),
                              ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream))
    _check(code, "sa_attn_sparse")
    return o, lse


def sa_attn_prepare(v: torch.Tensor, row_ptr: torch.Tensor, col_idx: torch.Tensor, *,
                    workspace: torch.Tensor, q_block: int = 64, qk_format="bf16",
                    dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """First half of sa_attn_sparse: V repacked into ``workspace`` and the
    tile pairs chosen from the route. Returns the workspace."""
    _require_cuda(v, row_ptr, col_idx, workspace)
    p = make_params(v, v, v, v, q_block=q_block, qk_format=qk_format)
    if workspace.numel() * workspace.element_size() < sa_attn_workspace_bytes(p):
        raise ValueError("workspace too small")
    code = load_library().sa_attn_prepare(ctypes.byref(p), _ptr(v), _ptr(row_ptr), _ptr(col_idx),
                                          _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _ptr(dev_status), _stream(stream))
    _check(code, "sa_attn_prepare")
    return workspace


def sa_attn_run(q: torch.Tensor, k: torch.Tensor, row_ptr: torch.Tensor, col_idx: torch.Tensor,
                scale: float = 0.0, *, workspace: torch.Tensor, v_like: Optional[torch.Tensor] = None,
                o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                want_lse: bool = True, q_block: int = 64, qk_format="bf16",
                dev_status: Optional[torch.Tensor] = None, stream=None):
    """Second half of sa_attn_sparse: the attention kernel over a workspace
    sa_attn_prepare filled (with 8-bit scores, after quantising q and k into
    it). ``v_like`` gives V's strides (default q's)."""
    _require_cuda(q, k, row_ptr, col_idx, workspace)
    o, lse = _attn_out(q, o, lse, want_lse)
    p = make_params(q, k, v_like, o, scale=scale, q_block=q_block, qk_format=qk_format)
    code = load_library().sa_attn_run(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(row_ptr),
                                      _ptr(col_idx), _ptr(o), _ptr(lse), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _ptr(dev_status), _stream(stream))
    _check(code, "sa_attn_run")
    return o, lse


def sa_qk_quantize(q: torch.Tensor, k: torch.Tensor, *,
                   dev_status: Optional[torch.Tensor] = None, stream=None):
    """The e4m3 codes of q and k (uint8 [B,S,H,D]) and the scale exponents of
    their 64-token blocks (int8 [B,H,Nb]); see sa.h."""
    _require_cuda(q, k)
    B, S, H, D = q.shape
    nb = (S + 63) // 64
    q8 = torch.empty((B, S, H, D), dtype=torch.uint8, device=q.device)
    k8 = torch.empty_like(q8)
    qe = torch.empty((B, H, nb), dtype=torch.int8, device=q.device)
    ke = torch.empty_like(qe)
    p = make_params(q, k)
    code = load_library().sa_qk_quantize(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(q8), _ptr(k8),
                                         _ptr(qe), _ptr(ke), _ptr(dev_status), _stream(stream))
    _check(code, "sa_qk_quantize")
    return q8, k8, qe, ke


def sa_attn_dense(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float = 0.0, *,
                  o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  want_lse: bool = True, workspace: Optional[torch.Tensor] = None,
                  qk_format="bf16", dev_status: Optional[torch.Tensor] = None, stream=None):
    """Attention over every key block (density 100%)."""
    _require_cuda(q, k, v)
    lib = load_library()
    o, lse = _attn_out(q, o, lse, want_lse)
    p = make_params(q, k, v, o, scale=scale, qk_format=qk_format)
    ws = _workspace(sa_attn_workspace_bytes(p), q.device, workspace)
    code = lib.sa_attn_dense(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
                             _stream(stream))
    _check(code, "sa_attn_dense")
    return o, lse


def sa_forward_host(q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor,
                    prefix_len: int, tau: float, scale: float = 0.0, *, bufs: dict,
                    mode="threshold", q_block: int = 64, o_host: Optional[torch.Tensor] = None,
                    lse_host: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One layer from (pinned) host tensors through the device buffers in
    ``bufs`` (q, k, v, o, lse, row_ptr, col_idx, ws, status); returns o_host.
    Enqueues only; synchronise the stream before reading o_host."""
    lib = load_library()
    if o_host is None:
        o_host = torch.empty_like(q_host, pin_memory=True)
    p = make_params(bufs["q"], prefix_len=prefix_len, tau=tau, scale=scale, mode=mode,
                    q_block=q_block)
    ws = bufs["ws"]
    code = lib.sa_forward_host(
        ctypes.byref(p), _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(o_host), _ptr(lse_host),
        _ptr(bufs["q"]), _ptr(bufs["k"]), _ptr(bufs["v"]), _ptr(bufs["o"]), _ptr(bufs.get("lse")),
        _ptr(bufs["row_ptr"]), _ptr(bufs["col_idx"]), bufs["col_idx"].numel(), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(bufs.get("status")), _stream(stream))
    _check(code, "sa_forward_host")
    return o_host


def alloc_layer_buffers(B: int, S: int, H: int, D: int, device="cuda", qk_format="bf16") -> dict:
    """Device buffers for sa_forward_host (one workspace sized for both calls)."""
    q = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=device)
    p = make_params(q, qk_format=qk_format)
    bufs = {"q": q, "k": torch.empty_like(q), "v": torch.empty_like(q), "o": torch.empty_like(q),
            "lse": torch.empty((B, H, S), dtype=torch.float32, device=device),
            "row_ptr": torch.empty(int(load_library().sa_route_rows(ctypes.byref(p))) + 1,
                                   dtype=torch.int32, device=device),
            "col_idx": torch.empty(sa_route_max_nnz(p), dtype=torch.int32, device=device),
            "status": torch.zeros(1, dtype=torch.int32, device=device)}
    nbytes = max(sa_route_workspace_bytes(p), sa_attn_workspace_bytes(p))
    bufs["ws"] = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return bufs


def check_dev_status(dev_status: torch.Tensor, what: str = "device status") -> None:
    """Raise if the kernels reported a device-side condition."""
    val = int(dev_status.item())
    if val:
        raise SaError(int(load_library().sa_dev_status_decode(val)), f"{what} (bits {val:#x})")
