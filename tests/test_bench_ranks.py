"""The replicas path of the benchmark with two ranks on CPU (gloo): each rank gets its own
batch (shifted data seed), the step time is the slowest rank's, and the rate counts every
rank's positions.  The benchmark's GPU runs use the same functions over NCCL."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.get("tiny")
        wr = bench.replica_workload(w, rank)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        first_u = float(workloads.generate(wr, requests=[0], with_T=False).U[0, 0, 0])
        q.put((rank, wr.seed, t, first_u))
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_is_the_slowest_rank_and_batches_differ():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, t0, u0), (r1, s1, t1, u1) = out
    assert (r0, r1) == (0, 1)
    assert t0 == t1 == 15.0                       # the max over ranks on every rank
    assert s0 != s1 and u0 != u1                  # independent batches


def test_whole_job_rate_counts_every_replica():
    w = workloads.get("qwen3_4b_like")
    one = bench.whole_job_rate(1, w, 0.2)
    assert one == pytest.approx(w.B * w.gamma / 0.2e-3)
    assert bench.whole_job_rate(4, w, 0.2) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) on the small
    workload: one JSON line with the metric, the reference marker, a cpu_baseline that
    describes the run, and an e2e entry with no host transfers."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == 3 and line["warmup"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny"
