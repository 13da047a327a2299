"""The N > 1 path of bench.py on the CPU: one process per rank over gloo.

The stage has no exchange step (dX is per token, dW is the caller's to
combine across ranks), so N GPUs run N independent replicas; what needs to be
right is the host logic around them: each replica draws its own inputs, every
rank ends up with the slowest rank's time, and the whole-job value counts the
bytes of all ranks over that time.  The reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from rms_backward_gb300 import workloads as WL
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                       # a slower rank 1
    slowest = bench._max_over_ranks(ms, world)
    seed = bench._replica_seed(WL.CONFIGS["tiny"]["seed"], rank)
    wl = WL.make("tiny", T=8, K=16, seed=seed)
    dist.barrier()
    out.put((rank, slowest, seed, wl.x.tobytes()))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time_and_draw_their_own_inputs():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get() for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (r0, s0, seed0, x0), (r1, s1, seed1, x1) = res
    assert s0 == s1 == 15.0                      # max over ranks, on every rank
    assert seed0 != seed1 and x0 != x1           # independent replicas


def test_aggregate_counts_every_rank_over_the_slowest_time():
    import bench
    assert bench._aggregate_gbs(1_000_000_000, 1, 1000.0) == pytest.approx(1.0)
    assert bench._aggregate_gbs(1_000_000_000, 4, 1000.0) == pytest.approx(4.0)
    assert bench._max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the bench's keys; a short time budget keeps this a CPU test."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--ref-seconds", "3"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    for key in ("metric", "value", "unit", "ms_per_step", "higher_is_better", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["sample_tokens_per_step"] >= 1
