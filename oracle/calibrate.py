"""Calibrate the synthetic-input constants against the oracle's block density.

Test infrastructure: it calls only ``oracle`` and the seeded generators in
``sa_inputs``. It prints the constants that ``sa_inputs`` commits:

* Tiny:    tau by bisection so that the block density is 25% (+-1%).
* Mid:     amplitude A by bisection for 20% density at tau = 1.0.
* Release: amplitude A by bisection for 19% density at tau = 1.0
           (the pages report 19.65% and 18.04% on the real activations).
* Long:    the Release amplitude at tau = 1.0; if the density falls outside
           12-15%, tau by bisection for 13.5%.

Run: ``python -m oracle.calibrate [tiny|mid|release|long ...]``.
"""

from __future__ import annotations

import sys
import time

import numpy as np

import sa_inputs
from . import sa_oracle as orc


def density_for(q, k, cfg, tau):
    r = orc.route_ref(q, k, cfg.P, tau)
    return orc.block_density(r["kept"])


def bisect(fn, lo, hi, target, iters=30, tol=2e-4, decreasing=True):
    """Find x in [lo, hi] with fn(x) ~= target for a monotone fn."""
    x = 0.5 * (lo + hi)
    for _ in range(iters):
        x = 0.5 * (lo + hi)
        d = fn(x)
        print(f"    x={x:.6f} density={d:.5f}", flush=True)
        if abs(d - target) < tol:
            break
        if (d > target) == decreasing:
            lo = x
        else:
            hi = x
    return x


def pooled_probs(q, k, cfg):
    qbar = orc.pool_blocks(orc.as_f64(q))
    kbar = orc.pool_blocks(orc.as_f64(k))
    return orc.pooled_softmax(orc.pooled_logits(qbar, kbar, cfg.scale))


def calibrate_tau(cfg, target):
    q, k, _ = sa_inputs.make_qkv(cfg)
    p = pooled_probs(q, k, cfg)

    def dens(tau):
        return orc.block_density(orc.select_blocks(p, tau, cfg.P))

    return bisect(dens, 0.5, 2.0, target)


def calibrate_amp(cfg, target, lo=0.0, hi=3.0):
    qn, kn, _, lr, (a, b) = sa_inputs.make_qkv(cfg, keep_parts=True)

    def dens(amp):
        q = sa_inputs.combine(qn, lr, a, b, amp)
        k = sa_inputs.combine(kn, lr, a, b, amp)
        return density_for(q, k, cfg, cfg.tau)

    return bisect(dens, lo, hi, target)


def main(names):
    for name in names:
        t0 = time.time()
        cfg = sa_inputs.get_config(name)
        if name == "tiny":
            x = calibrate_tau(cfg, 0.25)
            print(f"TINY_TAU = {x:.4f}")
        elif name == "mid":
            x = calibrate_amp(cfg, 0.20)
            print(f"MID_AMP = {x:.4f}")
        elif name == "release":
            x = calibrate_amp(cfg, 0.19)
            print(f"RELEASE_AMP = {x:.4f}")
        elif name == "long":
            q, k, _ = sa_inputs.make_qkv(cfg)
            p = pooled_probs(q, k, cfg)
            d1 = orc.block_density(orc.select_blocks(p, 1.0, cfg.P))
            print(f"    long density at tau=1.0: {d1:.5f}")
            if 0.12 <= d1 <= 0.15:
                print("LONG_TAU = 1.0")
            else:
                x = bisect(lambda t: orc.block_density(orc.select_blocks(p, t, cfg.P)),
                           0.25, 4.0, 0.135)
                print(f"LONG_TAU = {x:.4f}")
        print(f"  ({name}: {time.time() - t0:.1f} s)", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["tiny", "mid", "release", "long"])
