"""The benchmark's multi-rank host logic on CPU: two gloo ranks (replicas of
the workload, no data-path collective), the step time is the maximum over
ranks, the job value counts every rank's bytes, and the reference arm runs on
rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r measured (10 + r) ms per step, attention 5 * (r + 1), e2e 20 - r
    got = bench.max_over_ranks([10.0 + rank, 5.0 * (rank + 1), 20.0 - rank], world, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_and_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 10.0, 20.0]
    sys.path.insert(0, ROOT)
    import bench
    # two replicas of 1 GB each in the slowest rank's 11 ms
    assert bench.job_value(2, 10**9, 11.0) == pytest.approx(2e9 / 11e-3 / 1e9)
    assert bench.max_over_ranks([1.0, 2.0], 1, None) == [1.0, 2.0]


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
