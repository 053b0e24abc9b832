"""The N > 1 host logic of the benchmark on CPU: two gloo ranks, the token
data-parallel replicas' timing reduction (slowest rank wins) and whole-job
throughput (all ranks' tokens over that time).  No data-path collective exists
in the layer itself, so nothing else crosses ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 10.0 + 5.0 * rank           # rank 1 is the slow one
    got = bench.max_over_ranks(mine, world)
    val = bench.job_throughput(2048, 50, world, got)
    q.put((rank, got, val))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    # 2 ranks x 50 steps x 2048 tokens over 15 ms
    assert res[0][2] == pytest.approx(2 * 50 * 2048 / 0.015)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(16, 10, 1, 2.0) == pytest.approx(16 * 10 / 0.002)


def test_bench_gpus_flag_starts_that_many_ranks():
    # `bench.py --gpus 2` without a launcher starts two ranks itself
    # (torch.distributed.run on 127.0.0.1); with --launch-check they meet over
    # gloo on CPU, reduce their times (the slowest wins) and rank 0 prints
    # n_gpus = 2
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--launch-check"], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["max_ms"] == 11.0
