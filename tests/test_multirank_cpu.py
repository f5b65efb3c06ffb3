"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2): the path
shards into independent replicas (no exchange inside the mixers), so the
only cross-rank steps are the barrier and the max of the ranks' times; the
whole-job throughput is the sum over replicas at the slowest rank's time.
The reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(2.0 + 3.0 * rank, world, "cpu")  # rank 1 is the slow one
        q.put((rank, ms, bench.job_throughput(32, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [5.0, 5.0]  # every rank reports the slowest rank's time
    assert got[0][2] == pytest.approx(2 * 32 / 5e-3)  # two replicas of 32 nodes in 5 ms each


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.job_throughput(32, 1, 2.0) == pytest.approx(16000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:
        config, steps, warmup = 3, 1, 3
    bench.run_reference(A(), rank=1, world=2)  # returns at once, prints nothing
    assert capsys.readouterr().out == ""
