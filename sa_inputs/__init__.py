"""Seeded synthetic Q/K/V for the routed block-sparse self-attention layer.

This module only draws inputs. It holds none of the attention or routing
arithmetic, and both the CPU oracle side (tests, calibration, CPU baseline)
and the CUDA side (tests, benchmark) take their inputs from here.

The pages measure the layer on activations of a 33B audio-video diffusion
transformer ("MiniMax H3 runs on single 4090 with 4.44x speedup over dense
execution", third paragraph: tensor [1, 38247, 56, 128]; the Sol-Engine
H3-DataCenter release page, policy paragraph: 38,247 tokens per layer, a
951-token multimodal prefix, 1344x768 video with 124 frames). Those
activations are not available, so these generators stand in for them:

* ``tiny``    S=1,024, prefix 64, H=4, D=64: Q, K, V iid N(0,1).
* ``mid``     S=8,192, prefix 256, H=8, D=128: Q, K = 0.5*N(0,1) + A*phi(pos) W_h
              with a rank-8 1-D positional basis; V iid N(0,1).
* ``release`` S=38,247 = 951 prefix tokens (iid N(0,1)) + 37,296 grid tokens on a
              37x24x42 (T x Y x X) latent grid in t-major raster order, with
              Q, K = N(0,1) + A*phi(t,y,x) W_h (rank 12); V iid N(0,1).
* ``dense``   the release tensors, routed at 100% density.
* ``long``    S=112,640 = 951 prefix tokens + 110 full 24x42 frames + one partial
              frame of 809 tokens, same generator and amplitude as ``release``.

``W_h`` (shape [rank, D], entries N(0, 1/rank)) is shared by Q and K of head h,
so q.k grows as the positional distance shrinks, which makes routing favour
nearby blocks. Draw order from one seeded ``torch.Generator('cpu')``: Q noise,
K noise, V, then W. Values are drawn in fp32 and rounded once to bf16
(round-to-nearest-even).

For the QK-norm + RoPE prologue the module also draws the norm weights
(``qk_norm_weights``: gamma = 1 + 0.1 N(0,1), one vector for Q and one for K,
from their own seeded generator) and builds the rotary tables
(``rope_tables``: cos/sin of the angle of every token and pair, fp32
[S, D/2]; 1-D over the token index, or 3-D over (t, y, x) for the latent-grid
workloads with the prefix tokens along t). These are inputs of the kernel,
as the model's weights and positions would be.

The amplitudes ``A`` and the Tiny/Long ``tau`` values are calibration results
(bisection on the oracle's block density); the script that produced them is
``oracle/calibrate.py``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch

BLOCK = 64

# Calibrated constants (written by oracle/calibrate.py; targets in its header).
TINY_TAU = 1.0147
MID_AMP = 0.7991
RELEASE_AMP = 1.2100
LONG_TAU = 1.3047


@dataclass(frozen=True)
class Config:
    name: str
    S: int
    P: int
    H: int
    D: int
    tau: float
    kind: str  # 'iid' | 'pos1d' | 'grid3d'
    noise: float = 1.0
    amp: float = 0.0
    grid: Tuple[int, int, int] = (0, 0, 0)  # (T, Y, X) of the latent grid
    t_period: int = 37  # temporal period of the grid basis, in frames
    dense: bool = False
    B: int = 1
    seed: int = 0

    @property
    def Nb(self) -> int:
        return (self.S + BLOCK - 1) // BLOCK

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


CONFIGS = {
    "tiny": Config("tiny", S=1024, P=64, H=4, D=64, tau=TINY_TAU, kind="iid"),
    "mid": Config("mid", S=8192, P=256, H=8, D=128, tau=1.0, kind="pos1d",
                  noise=0.5, amp=MID_AMP),
    "release": Config("release", S=38247, P=951, H=56, D=128, tau=1.0,
                      kind="grid3d", amp=RELEASE_AMP, grid=(37, 24, 42)),
    "dense": Config("dense", S=38247, P=951, H=56, D=128, tau=0.0,
                    kind="grid3d", amp=RELEASE_AMP, grid=(37, 24, 42), dense=True),
    "long": Config("long", S=112640, P=951, H=56, D=128, tau=LONG_TAU,
                   kind="grid3d", amp=RELEASE_AMP, grid=(111, 24, 42)),
}


def get_config(name: str, **overrides) -> Config:
    cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg


def positional_basis(cfg: Config, n_tokens: int) -> torch.Tensor:
    """Low-rank positional features phi for the non-prefix tokens, fp32 [n, rank].

    pos1d: {cos, sin}(2*pi*f*pos/S) for f in {1, 2, 4, 8} (rank 8), pos = token index.
    grid3d: {cos, sin}(2*pi*f*c/L) for f in {1, 2} on each of the t, y, x axes
    (rank 12); L is the axis length for y and x and ``t_period`` frames for t,
    so a longer clip keeps the same per-frame frequencies.
    """
    if cfg.kind == "pos1d":
        pos = torch.arange(n_tokens, dtype=torch.float64) + cfg.P
        feats = []
        for f in (1, 2, 4, 8):
            ang = 2.0 * math.pi * f * pos / cfg.S
            feats += [torch.cos(ang), torch.sin(ang)]
        return torch.stack(feats, dim=1).float()
    if cfg.kind == "grid3d":
        _, Y, X = cfg.grid
        idx = torch.arange(n_tokens, dtype=torch.int64)
        t = (idx // (Y * X)).double()
        y = ((idx // X) % Y).double()
        x = (idx % X).double()
        feats = []
        for coord, L in ((t, cfg.t_period), (y, Y), (x, X)):
            for f in (1, 2):
                ang = 2.0 * math.pi * f * coord / L
                feats += [torch.cos(ang), torch.sin(ang)]
        return torch.stack(feats, dim=1).float()
    raise ValueError(f"no positional basis for kind {cfg.kind!r}")


def _structured_span(cfg: Config) -> Tuple[int, int]:
    """Token range [lo, hi) that carries the low-rank component."""
    if cfg.kind == "pos1d":
        return 0, cfg.S
    if cfg.kind == "grid3d":
        return cfg.P, cfg.S
    return 0, 0


def make_qkv(cfg: Config, seed: Optional[int] = None, amp: Optional[float] = None,
             keep_parts: bool = False):
    """Draw bf16 Q, K, V of shape [B, S, H, D] (contiguous, CPU).

    With ``keep_parts`` it also returns the fp32 pieces (noise and low-rank
    term) so a calibration loop can re-round Q/K for another amplitude without
    drawing again.
    """
    seed = cfg.seed if seed is None else seed
    amp = cfg.amp if amp is None else amp
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (cfg.B, cfg.S, cfg.H, cfg.D)
    qn = torch.randn(shape, generator=g, dtype=torch.float32)
    kn = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    lo, hi = _structured_span(cfg)
    lr = None
    if hi > lo:
        rank = 8 if cfg.kind == "pos1d" else 12
        w = torch.randn((cfg.H, rank, cfg.D), generator=g, dtype=torch.float32)
        w.mul_(1.0 / math.sqrt(rank))
        phi = positional_basis(cfg, hi - lo)  # [n, rank]
        lr = torch.einsum("nr,hrd->nhd", phi, w)  # [n, H, D]
    if cfg.noise != 1.0:
        qn.mul_(cfg.noise)
        kn.mul_(cfg.noise)
    if keep_parts:
        return qn, kn, v, lr, (lo, hi)
    q = combine(qn, lr, lo, hi, amp)
    del qn
    k = combine(kn, lr, lo, hi, amp)
    return q, k, v


def combine(noise: torch.Tensor, lr: Optional[torch.Tensor], lo: int, hi: int,
            amp: float) -> torch.Tensor:
    """noise + amp * low-rank term on tokens [lo, hi), rounded once to bf16."""
    out = noise.clone() if lr is not None and amp != 0.0 else noise
    if lr is not None and amp != 0.0:
        out[:, lo:hi].add_(lr.unsqueeze(0), alpha=amp)
    return out.to(torch.bfloat16)


def make_inputs(name: str, seed: Optional[int] = None):
    """Config plus its bf16 Q, K, V."""
    cfg = get_config(name)
    q, k, v = make_qkv(cfg, seed=seed)
    return cfg, q, k, v


def random_small(S: int, H: int, D: int, seed: int, B: int = 1, std: float = 1.0):
    """iid N(0, std^2) bf16 Q, K, V of shape [B, S, H, D] for edge-case tests."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, S, H, D)
    return tuple((torch.randn(shape, generator=g) * std).to(torch.bfloat16)
                 for _ in range(3))


def qk_norm_weights(D: int, seed: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """QK-norm weights gamma_q, gamma_k: fp32 [D] each, 1 + 0.1 N(0,1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 + seed)
    return tuple((1.0 + 0.1 * torch.randn(D, generator=g)).float() for _ in range(2))


def rope_tables(cfg: Config, base: float = 10000.0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Rotary tables cos, sin: fp32 [S, D/2] (pair i of token t turns by theta[t, i]).

    1-D (iid, pos1d): theta = t * base^(-2i/D) over the token index t.
    3-D (grid3d): the D/2 pairs split into t, y, x sections (the y and x
    sections D/12 pairs each, rounded down; t the rest); within a section of
    n pairs, pair j turns by pos * base^(-j/n), pos the token's coordinate on
    that axis. Prefix token j sits at t = j, y = x = 0; grid token (f, y, x)
    at t = P + f.
    """
    S, D = cfg.S, cfg.D
    half = D // 2
    if cfg.kind != "grid3d":
        t = torch.arange(S, dtype=torch.float64)[:, None]
        w = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)
        ang = t * w[None, :]
    else:
        _, Y, X = cfg.grid
        n_y = n_x = D // 12
        n_t = half - n_y - n_x
        idx = torch.arange(S, dtype=torch.int64)
        g = (idx - cfg.P).clamp(min=0)
        pre = idx < cfg.P
        tpos = torch.where(pre, idx, cfg.P + g // (Y * X)).double()
        ypos = torch.where(pre, torch.zeros_like(idx), (g // X) % Y).double()
        xpos = torch.where(pre, torch.zeros_like(idx), g % X).double()
        cols = []
        for pos, n in ((tpos, n_t), (ypos, n_y), (xpos, n_x)):
            w = base ** (-torch.arange(n, dtype=torch.float64) / n)
            cols.append(pos[:, None] * w[None, :])
        ang = torch.cat(cols, dim=1)
    return torch.cos(ang).float().contiguous(), torch.sin(ang).float().contiguous()
