"""Benchmark of one routed block-sparse attention layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload release|long|dense|mid|tiny] [--route-mode M] [--tau T]
                    [--q-block 64|128] [--prologue] [--no-e2e] [--no-cpu]

One step = the whole hot path on one batch of synthetic input already in
HBM: sa_route (pool, score, select, recheck, scan, emit) then sa_attn_sparse
as its two halves (sa_attn_prepare: V repack and tile pairing; sa_attn_run:
the attention kernel, timed on its own for the roofline), at the release
shape S=38,247, H=56, D=128, prefix 951, tau=1.0 (~19% block density). The metric is effective TFLOP/s on the
routed pairs: FLOPs = 4 * D * sum over routed (query block, key block) pairs
of (valid queries) x (valid keys), divided by the step time.

Inputs (Q, K, V, O = 2.19 GB) are larger than the 129 MB L2, so no flush runs
between steps. Steps are timed with CUDA events on the stream the kernels are
launched on, W untimed warm-up steps first, with a barrier and
torch.cuda.synchronize() on both sides; for N > 1 each rank (one GPU each,
torchrun) runs an independent replica of the layer (the path has no exchange
step) and the max time over ranks is used.

--prologue adds the QK-norm + RoPE step in front (sa_qk_prologue on the
workload's Q, K taken as the pre-norm projections, with seeded norm weights
and the workload's rotary tables), which also pools Q and K for the router
(sa_route_pooled replaces sa_route's own pooling pass).

--impl reference times the CPU oracle (the reference arm: no code exists to
run for this method) on a bounded sample of the same workload and scales it
to a whole layer.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import sa_inputs  # noqa: E402

METRIC = "ms/layer and effective TFLOP/s (% of GB300 bf16 peak) at S=38,247, ~18% density"
UNIT = "TFLOP/s"
# our kernels per step: the router (pool, score, select, recheck, scan, emit),
# then the tile pairing (pair_rank, pair_match; only for 64-token query blocks
# when there are more than two of them), the V repack and the attention
# kernel; dense mode runs just the last two
ROUTE_KERNELS, PAIR_KERNELS, ATTN_KERNELS = 6, 2, 2

# DRAM traffic of one attention-kernel launch at the release workload, from
# the ncu capture summarised under profiles/ (taken with 8 of the 56 heads and
# scaled by 7: the traffic grows with the heads processed), valid only for the
# attn.cu it was taken on (sha256 prefix); otherwise reported as null.
ATTN_TRAFFIC = {"bytes": 2.166e9, "attn_cu_sha256": "305b8aca01342ac8"}


def file_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# ---------------------------------------------------------------- helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_tflops(flops_per_rank: int, ms_per_step: float, world: int) -> float:
    """Aggregate throughput of ``world`` replicas that each process
    ``flops_per_rank`` per step, timed by the slowest rank (``ms_per_step`` is
    already the max over ranks)."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def timed_max_ms(local_ms: float, steps: int, world: int, device=None) -> float:
    """Per-step time of the job: the slowest rank's timed region / steps."""
    return reduce_max(local_ms, world, device) / steps


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[1].isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = sorted({self.REASONS[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        sm = [int(r[1]) for r in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return 0.0

        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]),
                "power_w_max": max(num(r[3]) for r in rows), "samples": len(rows),
                "reasons": reasons}


# ------------------------------------------------------------- our arm -----

def routed_flops(row_ptr: np.ndarray, col_idx: np.ndarray, B, H, S, D) -> int:
    """4 * D * sum over routed pairs of valid queries x valid keys."""
    Nb = (S + 63) // 64
    counts = np.minimum(64, S - 64 * np.arange(Nb))
    cs = np.concatenate([[0], np.cumsum(counts[col_idx])])
    per_row = cs[row_ptr[1:]] - cs[row_ptr[:-1]]
    ni = counts[np.arange(B * H * Nb) % Nb]
    return int(4 * D * int((ni * per_row).sum()))


def run_ours(args):
    import block_sparse_attention_sa_gb300 as sa
    from block_sparse_attention_sa_gb300 import build as _build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    barrier(world)
    sa.load_library()

    cfg = sa_inputs.get_config(args.workload, **({"H": args.heads} if args.heads else {}))
    tau = cfg.tau if args.tau is None else args.tau
    mode, qblk = args.route_mode, args.q_block
    q, k, v = sa_inputs.make_qkv(cfg)
    B, S, H, D = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    f8 = args.qk_format == "fp8"
    bufs = sa.alloc_layer_buffers(B, S, H, D, device=dev, qk_format=args.qk_format)
    ws, status = bufs["ws"], bufs["status"]
    o, lse, rp_buf, ci_buf = bufs["o"], bufs["lse"], bufs["row_ptr"], bufs["col_idx"]
    stream = torch.cuda.current_stream(dev)
    dense = cfg.dense
    pro = args.prologue and not dense
    if pro:
        gq, gk = (t.to(dev) for t in sa_inputs.qk_norm_weights(D))
        cos, sin = (t.to(dev) for t in sa_inputs.rope_tables(cfg))
        qn, kn = torch.empty_like(qd), torch.empty_like(kd)   # the prologue's outputs

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        qa, ka = qd, kd
        if pro:
            sa.sa_qk_prologue(qd, kd, gq, gk, 1e-6, cos, sin, q_block=qblk, q_out=qn, k_out=kn,
                              workspace=ws, dev_status=status)
            qa, ka = qn, kn
        if ev is not None:
            ev[1].record(stream)
        if pro:
            sa.sa_route_pooled(qa, ws, cfg.P, tau, k=ka, mode=mode, q_block=qblk, row_ptr=rp_buf,
                               col_idx=ci_buf, dev_status=status)
        elif not dense:
            sa.sa_route(qa, ka, cfg.P, tau, mode=mode, q_block=qblk, row_ptr=rp_buf,
                        col_idx=ci_buf, workspace=ws, dev_status=status)
        if ev is not None:
            ev[2].record(stream)
        if dense:
            sa.sa_attn_dense(qa, ka, vd, o=o, lse=lse, workspace=ws, qk_format=args.qk_format,
                             dev_status=status)
            if ev is not None:
                ev[3].record(stream)
        else:
            # sa_attn_sparse as its two halves, so that the attention kernel
            # (the dominant one) is timed on its own
            sa.sa_attn_prepare(vd, rp_buf, ci_buf, workspace=ws, q_block=qblk,
                               qk_format=args.qk_format, dev_status=status)
            if ev is not None:
                ev[3].record(stream)
            sa.sa_attn_run(qa, ka, rp_buf, ci_buf, workspace=ws, v_like=vd, o=o, lse=lse,
                           q_block=qblk, qk_format=args.qk_format, dev_status=status)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sa.check_dev_status(status, "bench warm-up")
    Nb = cfg.Nb
    if dense:
        row_ptr = np.arange(B * H * Nb + 1, dtype=np.int64) * Nb
        col_idx = np.tile(np.arange(Nb), B * H * Nb)
    else:
        row_ptr = rp_buf.cpu().numpy().astype(np.int64)
        col_idx = ci_buf[: int(row_ptr[-1])].cpu().numpy().astype(np.int64)
    flops = routed_flops(row_ptr, col_idx, B, H, S, D)
    density = float(row_ptr[-1]) / (B * H * Nb * Nb)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    sa.check_dev_status(status, "bench")
    ms_step = timed_max_ms(start.elapsed_time(end), args.steps, world, dev)
    total_ms = ms_step * args.steps
    pro_ms = [e[0].elapsed_time(e[1]) for e in evs]
    route_ms = [e[1].elapsed_time(e[2]) for e in evs]
    attn_ms = [e[2].elapsed_time(e[4]) for e in evs]          # the attention call
    kern_ms = [e[3].elapsed_time(e[4]) for e in evs]          # the attention kernel
    # (dense: sa_attn_dense as one call, so the kernel time is the call's)
    value = whole_job_tflops(flops, ms_step, world)
    attn_avg = statistics.mean(attn_ms)
    kern_avg = attn_avg if dense else statistics.mean(kern_ms)
    burst, sustained, _, peak_src = measured_peaks()
    long_region = total_ms > 1000.0
    peak = sustained if long_region else burst
    if f8:
        # half the FLOPs (Q.K^T) at the e4m3 rate, nominally twice bf16's, half
        # (P.V) at the 16-bit rate: the mix's peak is 1 / (0.5/2 + 0.5) = 4/3 of bf16
        peak = round(peak * 4.0 / 3.0, 1)
    achieved = flops / (kern_avg * 1e-3) / 1e12
    call_achieved = flops / (attn_avg * 1e-3) / 1e12
    sha = file_sha(os.path.join(ROOT, "block_sparse_attention_sa_gb300", "csrc", "attn.cu"))
    # the counter was taken on the release workload with 64-token query blocks
    # (and the pairing's tile list): another workload or tile list has no number
    traffic = (ATTN_TRAFFIC["bytes"]
               if ATTN_TRAFFIC["attn_cu_sha256"] and sha.startswith(ATTN_TRAFFIC["attn_cu_sha256"])
               and cfg.name == "release" and H == 56 and qblk == 64 and not dense and not pro
               and not f8 else None)

    e2e = None if (args.no_e2e or pro or f8) else run_e2e(sa, cfg, q, k, v, bufs, flops, args, world, dev,
                                           stream, tau, mode, qblk)
    pairing = Nb > 2 and qblk == 64
    per_step = (ATTN_KERNELS + (1 if f8 else 0)
                + (0 if dense else ROUTE_KERNELS + (PAIR_KERNELS if pairing else 0)))

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the arithmetic of the path: Q.K^T operands, P.V operands, accumulation
        "dtype": ("e4m3 QK, fp16 PV, fp32 accumulate" if f8
                  else "bf16 QK, fp16 PV, fp32 accumulate"),
        "data": "synthetic (seeded; stands in for the model's activations)",
        "config": {"workload": cfg.name, "B": B, "S": S, "H": H, "D": D, "prefix": cfg.P,
                   "tau": tau, "route_mode": "dense" if dense else mode, "block": 64,
                   "q_block": qblk, "qk_format": args.qk_format,
                   "density": round(density, 5),
                   "routed_tflop_per_layer": round(flops / 1e12, 4),
                   "ms_route": round(statistics.mean(route_ms), 4),
                   **({"prologue": "QK-norm + RoPE, pooling fused (sa_qk_prologue)",
                       "ms_prologue": round(statistics.mean(pro_ms), 4),
                       # read Q, K and write them back: 4 x S x H x D x 2 bytes
                       "prologue_gbs": round(4 * q.numel() * 2 / (statistics.mean(pro_ms) * 1e-3)
                                             / 1e9, 1)} if pro else {}),
                   "ms_attn": round(attn_avg, 4),
                   "ms_attn_kernel": round(kern_avg, 4),
                   "attn_call_frac": round(call_achieved / peak, 4),
                   "l2": "inputs larger than L2 (Q/K/V/O %.2f GB), no flush" % (4 * q.numel() * 2 / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor",
                     "kernel": ("attn_fwd_kernel (V repack included: sa_attn_dense is one call)"
                                if dense else "attn_fwd_kernel"),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_kind": (f"{'sustained' if long_region else 'burst'} bf16, {peak_src}"
                                   + (", x 4/3 for e4m3 Q.K^T + fp16 P.V (nominal e4m3 rate 2x bf16)"
                                      if f8 else "")),
                     "traffic": traffic},
        "gpu_launches": per_step * args.steps,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu and rank == 0:
        # the oracle times the whole layer where it finishes in about a minute
        # (tiny, mid), else a bounded sample scaled to the layer
        result["cpu_baseline"] = cpu_baseline(cfg, q, k, v, flops, budget_s=15.0, tau=tau,
                                              mode=mode, q_block=qblk,
                                              full_layer=cfg.name in ("tiny", "mid") and not f8)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(sa, cfg, q, k, v, bufs, flops, args, world, dev, stream, tau, mode, qblk):
    """The same layer through sa_forward_host: pinned host Q/K/V in, host O out,
    copies inside the timed region."""
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh, pin_memory=True)
    steps = max(5, min(args.steps, 10))
    for _ in range(2):
        sa.sa_forward_host(qh, kh, vh, cfg.P, tau, bufs=bufs, mode=mode, q_block=qblk,
                           o_host=oh)
    torch.cuda.synchronize()
    # each call starts after the previous one has finished (its copies back
    # included), so an event pair per call times it exactly; the host link is
    # shared with the machine's other GPUs, so the median call is reported
    # (the mean beside it)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s_ev, e_ev in evs:
        s_ev.record(stream)
        sa.sa_forward_host(qh, kh, vh, cfg.P, tau, bufs=bufs, mode=mode, q_block=qblk,
                           o_host=oh)
        e_ev.record(stream)
    torch.cuda.synchronize()
    per = [s_ev.elapsed_time(e_ev) for s_ev, e_ev in evs]
    ms = reduce_max(statistics.median(per), world, dev)
    mean = reduce_max(statistics.mean(per), world, dev)
    nbytes = q.numel() * 2
    return {"value": round(whole_job_tflops(flops, ms, world), 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "ms_per_step_mean": round(mean, 4),
            "timing": f"median of {steps} calls", "h2d_bytes_per_step": 3 * nbytes,
            "d2h_bytes_per_step": nbytes}


# ------------------------------------------------------- the CPU oracle ----

def blas_threads():
    """(threads, how) of the BLAS numpy calls: threadpoolctl's report where it
    is installed, else the thread-count variables, else None."""
    try:
        from threadpoolctl import threadpool_info
        n = [d["num_threads"] for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n)), "threadpoolctl"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var]), var
    return None, "not reported by the BLAS (its default is one thread per core)"


def cpu_baseline(cfg, q, k, v, flops, budget_s=15.0, seed=0, tau=None, mode="threshold",
                 q_block=64, full_layer=False):
    """Time the oracle on the layer. With ``full_layer`` the whole layer (every
    head routed and attended); otherwise a bounded sample scaled to a whole
    layer: the route of one head in full, plus as many query blocks of that
    head as fit in ``budget_s`` (at least 4), extrapolated linearly to all
    heads and blocks."""
    import oracle

    B, S, H, D = q.shape
    Nb = cfg.Nb
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads, how = blas_threads()
    tau = cfg.tau if tau is None else tau
    if full_layer:
        t0 = time.perf_counter()
        r = oracle.route_ref(q, k, cfg.P, float(np.float32(tau)), mode=mode, q_block=q_block)
        t_route = time.perf_counter() - t0
        oracle.attn_ref(q, k, v, r["row_ptr"], r["col_idx"])
        layer_s = time.perf_counter() - t0
        return {"value": round(flops / layer_s / 1e12, 6), "unit": UNIT, "cores": cores,
                "threads": threads, "threads_source": how, "kind": "oracle",
                "timing": "the full layer, timed once",
                "sample": f"the full layer: {B * H} heads routed ({t_route:.1f} s) and "
                          f"attended, {layer_s:.1f} s"}
    h = seed % H
    qs, ks, vs = (t[:, :, h:h + 1].contiguous() for t in (q, k, v))
    t0 = time.perf_counter()
    r = oracle.route_ref(qs, ks, cfg.P, float(np.float32(tau)), mode=mode, q_block=q_block)
    t_route = time.perf_counter() - t0
    order = np.random.default_rng(seed).permutation(Nb)
    t_attn, n_done = 0.0, 0
    while n_done < Nb and (n_done < 4 or t_attn < budget_s):
        i = int(order[n_done])
        t0 = time.perf_counter()
        oracle.attn_ref(qs, ks, vs, r["row_ptr"], r["col_idx"], items=[(0, 0, i)])
        t_attn += time.perf_counter() - t0
        n_done += 1
    layer_s = t_route * B * H + t_attn * (B * H * Nb / n_done)
    return {"value": round(flops / layer_s / 1e12, 6), "unit": UNIT, "cores": cores,
            "threads": threads, "threads_source": how, "kind": "oracle",
            "timing": "extrapolated from a sample",
            "sampled_s": round(t_route + t_attn, 2),
            "sample": f"head {h}: full route ({t_route:.1f} s) + {n_done} query blocks of "
                      f"attention ({t_attn:.1f} s); extrapolated linearly to {B * H} heads x "
                      f"{Nb} blocks = {layer_s:.0f} s per layer"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = sa_inputs.get_config(args.workload)
    tau = cfg.tau if args.tau is None else args.tau
    mode, qblk = args.route_mode, args.q_block
    q, k, v = sa_inputs.make_qkv(cfg)
    B, S, H, D = q.shape
    import oracle
    # the layer's routed FLOPs from the oracle's own route
    ref = oracle.route_ref(q, k, cfg.P, float(np.float32(tau)), mode=mode, q_block=qblk)
    flops = routed_flops(ref["row_ptr"], ref["col_idx"], B, H, S, D)
    del ref
    for w in range(args.warmup):
        cpu_baseline(cfg, q, k, v, flops, budget_s=1.0, seed=w, tau=tau, mode=mode,
                     q_block=qblk)
    vals = [cpu_baseline(cfg, q, k, v, flops, budget_s=5.0, seed=100 + s, tau=tau, mode=mode,
                         q_block=qblk) for s in range(args.steps)]
    value = statistics.mean(c["value"] for c in vals)
    ms = flops / (value * 1e12) * 1e3
    sampled = statistics.mean(c["sampled_s"] for c in vals)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 1), "higher_is_better": True, "scaling": "weak",
        "timing": (f"extrapolated from a sample: each of the {args.steps} steps times "
                   f"{sampled:.1f} s of the oracle (one head routed in full and a sample of its "
                   f"query blocks attended) and scales it linearly to the whole layer; "
                   f"ms_per_step is that extrapolated layer time, not a step's wall time"),
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "B": B, "S": S, "H": H, "D": D, "prefix": cfg.P,
                   "tau": tau, "route_mode": mode, "q_block": qblk},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": vals[0]["cores"],
                         "threads": vals[0]["threads"],
                         "threads_source": vals[0]["threads_source"], "kind": "oracle",
                         "timing": "extrapolated from a sample", "sample": vals[-1]["sample"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="release", choices=sorted(sa_inputs.CONFIGS))
    ap.add_argument("--heads", type=int, default=0,
                    help="override H (smaller captures for profiling)")
    ap.add_argument("--route-mode", default="threshold",
                    choices=["threshold", "dense_prefix_queries", "top_mass"],
                    help="reading of the router rule (sa.h SA_ROUTE_*)")
    ap.add_argument("--tau", type=float, default=None, help="override the workload's tau")
    ap.add_argument("--q-block", type=int, default=64, choices=[64, 128],
                    help="query block of the route (128: two key blocks per query block)")
    ap.add_argument("--qk-format", default="bf16", choices=["bf16", "fp8"],
                    help="arithmetic of the score product Q.K^T (fp8: 8-bit e4m3 scores)")
    ap.add_argument("--prologue", action="store_true",
                    help="QK-norm + RoPE in front, with the router's pooling fused in")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
