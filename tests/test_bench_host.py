"""bench.py's host-side arithmetic on CPU: the routed-FLOP count against the
oracle's, and the clock sampler's parsing of nvidia-smi lines (the throttle
reasons a run must report)."""

import os
import sys
import tempfile

import numpy as np

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_routed_flops_match_the_oracle():
    rng = np.random.default_rng(3)
    for S, H, D in ((1000, 2, 64), (38247 // 8, 3, 128), (65, 1, 128)):
        Nb = oracle.num_blocks(S)
        kept = rng.random((1, H, Nb, Nb)) < 0.3
        rp, ci = oracle.to_csr(kept)
        assert bench.routed_flops(rp, ci, 1, H, S, D) == oracle.routed_flops(rp, ci, 1, H, S, D)


def test_release_dense_flops():
    S, H, D = 38247, 56, 128
    Nb = oracle.num_blocks(S)
    rp, ci = oracle.dense_csr(1, H, S)
    assert bench.routed_flops(rp, ci, 1, H, S, D) == 4 * D * H * S * S   # 41.94 TFLOP


def _summary(lines):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    return c.summary()


def test_clock_summary_reports_reasons_and_median():
    idle = "0, 2070, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    cap = "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    hot = "0, 1500, 2070, 1400.0, 0x20, Not Active, Not Active, Active, Not Active"
    s = _summary([idle, cap, cap, hot, "garbage line"])
    assert s["samples"] == 4 and s["sm_max_mhz"] == 2070
    assert s["sm_mhz"] == (1980 + 1980) / 2                      # median of 4 samples
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert s["power_w_max"] == 1400.0
    assert _summary(["nothing"])["reasons"] == ["unsampled"]


def test_whole_job_value_and_max_over_ranks_single_rank():
    assert bench.timed_max_ms(100.0, 20, 1) == 5.0
    assert abs(bench.whole_job_tflops(8_000_000_000_000, 8.0, 1) - 1000.0) < 1e-9
