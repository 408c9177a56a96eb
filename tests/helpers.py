"""Shared helpers of the parity tests: build/load the library, run the CUDA
path through the binding, and compare with the oracle.

Tolerances (attention outputs, bf16):
* L2-relative error <= 1e-3 against the oracle's fp64 result rounded once to
  bf16, i.e. both sides in the output's precision. Rounding the exact result
  itself to bf16 already costs ~1.7e-3 L2-relative (the RMS relative error of
  round-to-nearest with an 8-bit significand), so a bound of 1e-3 can only be
  stated between two bf16 results.
* max-abs <= 3e-2 against the fp64 result.
* LSE (fp32) within 1e-3 + 1e-4 |lse| of the fp64 log-sum-exp.
Routing: identical kept sets except on oracle ties (|p Nb / tau - 1| <= 1e-6).
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle

L2_TOL = 1e-3
MAXABS_TOL = 3e-2


def lib():
    from block_sparse_attention_sa_gb300 import build as _build
    _build.build()
    import block_sparse_attention_sa_gb300 as sa
    sa.load_library()
    return sa


def f32(x: float) -> float:
    """The fp32 value the C ABI receives for a Python float."""
    return float(np.float32(x))


def kept_from_csr(row_ptr: np.ndarray, col_idx: np.ndarray, B: int, H: int, Nb: int) -> np.ndarray:
    kept = np.zeros((B * H * Nb, Nb), dtype=bool)
    for r in range(B * H * Nb):
        kept[r, col_idx[row_ptr[r]:row_ptr[r + 1]]] = True
    return kept.reshape(B, H, Nb, Nb)


def check_csr_wellformed(row_ptr: np.ndarray, col_idx: np.ndarray, Nb: int) -> None:
    assert row_ptr[0] == 0
    assert np.all(np.diff(row_ptr) >= 0)
    for r in range(len(row_ptr) - 1):
        cols = col_idx[row_ptr[r]:row_ptr[r + 1]]
        assert np.all(np.diff(cols) > 0), f"row {r} not ascending"
        assert cols.size == 0 or (cols[0] >= 0 and cols[-1] < Nb)


def compare_route(gpu_rp, gpu_ci, ref, B, H, Nb):
    """Returns (n_mismatch_outside_ties, n_ties)."""
    check_csr_wellformed(gpu_rp, gpu_ci, Nb)
    kept_gpu = kept_from_csr(gpu_rp, gpu_ci, B, H, Nb)
    ties = ref["ties"]
    diff = (kept_gpu != ref["kept"]) & ~ties
    return int(diff.sum()), int(ties.sum())


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def out_errors(o_gpu: np.ndarray, o_ref: np.ndarray):
    """(L2-rel vs bf16-rounded oracle, max-abs vs fp64 oracle, L2-rel vs fp64)."""
    ref_b = bf16_round(o_ref)
    den = np.linalg.norm(ref_b)
    l2 = np.linalg.norm(o_gpu - ref_b) / den if den > 0 else np.linalg.norm(o_gpu)
    den64 = np.linalg.norm(o_ref)
    l2_64 = np.linalg.norm(o_gpu - o_ref) / den64 if den64 > 0 else np.linalg.norm(o_gpu)
    return float(l2), float(np.abs(o_gpu - o_ref).max()) if o_ref.size else 0.0, float(l2_64)


def lse_ok(lse_gpu: np.ndarray, lse_ref: np.ndarray) -> bool:
    both_inf = np.isneginf(lse_gpu) & np.isneginf(lse_ref)
    fin = ~both_inf
    err = np.abs(lse_gpu[fin] - lse_ref[fin])
    return bool(np.all(err <= 1e-3 + 1e-4 * np.abs(lse_ref[fin])))


def sample_items(B: int, H: int, Nb: int, n_heads: int, n_blocks: int, seed: int,
                 must=(0,)):
    """Seeded (b, h, i) sample: n_heads heads x n_blocks query blocks, always
    including the blocks in ``must`` (e.g. first, prefix boundary, tail)."""
    rng = np.random.default_rng(seed)
    heads = sorted(rng.choice(H, size=min(n_heads, H), replace=False).tolist())
    items = []
    for b in range(B):
        for h in heads:
            forced = [i for i in must if 0 <= i < Nb]
            rest = [i for i in range(Nb) if i not in forced]
            extra = rng.choice(rest, size=max(0, min(n_blocks - len(forced), len(rest))),
                               replace=False).tolist()
            items += [(b, h, i) for i in sorted(set(forced + extra))]
    return items


def gather_rows(o: np.ndarray, lse: np.ndarray, items, S: int):
    """Concatenate the rows of the sampled query blocks (O [n, D], LSE [n])."""
    os_, ls_ = [], []
    for (b, h, i) in items:
        t0, t1 = 64 * i, min(S, 64 * i + 64)
        os_.append(o[b, t0:t1, h, :])
        ls_.append(lse[b, h, t0:t1])
    return np.concatenate(os_), np.concatenate(ls_)


def ref_rows(ref_items: dict, items):
    return (np.concatenate([ref_items[it][0] for it in items]),
            np.concatenate([ref_items[it][1] for it in items]))


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().double().numpy() if t.is_floating_point() else t.detach().cpu().numpy()
