"""bench.py's multi-rank host logic on CPU, world size 2 over gloo.

The layer has no exchange step, so N > 1 runs N independent replicas: each
rank times its own steps, the job's step time is the slowest rank's, and the
reported value is the work of all ranks over that time. These tests drive
exactly those helpers from two real processes (the GPU work itself is not
involved), and launch the reference arm under torchrun to check that only
rank 0 prints its line.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        # rank r "timed" 5 steps in 40 * (r + 1) ms: the slower rank sets the pace
        ms = bench.timed_max_ms(40.0 * (r + 1), 5, w)
        bench.barrier(w)
        val = bench.whole_job_tflops(3 * 10 ** 12, ms, w)
        out.put({"rank": r, "world": w, "local": local, "ms": ms, "value": val})
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in res] == [0, 1]
    assert all(d["world"] == 2 for d in res)
    assert [d["local"] for d in res] == [0, 1]
    # max over ranks of 40 ms and 80 ms, over 5 steps
    assert all(d["ms"] == pytest.approx(16.0) for d in res)
    # two replicas x 3 TFLOP each per 16 ms step = 375 TFLOP/s
    assert all(d["value"] == pytest.approx(375.0) for d in res)


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(7.5, 1) == 7.5
    assert bench.timed_max_ms(30.0, 3, 1) == pytest.approx(10.0)
    assert bench.whole_job_tflops(2 * 10 ** 12, 4.0, 1) == pytest.approx(500.0)
    bench.barrier(1)  # no process group needed


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1",
           "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
