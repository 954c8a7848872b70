"""bench.py's N > 1 path on the CPU: world_size-2 gloo ranks, each an
independent replica, combined as every replica's steps over the slowest
rank's time (the method has no exchange between replicas)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total, value = bench.replica_throughput(local_ms[rank], 10, world, dist, "cpu")
        e2e = bench.max_over_ranks(local_ms[rank] / 2, dist, "cpu")
        out.put((rank, total, value, e2e))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local = [100.0, 150.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, local, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value, e2e in got:
        assert total == 150.0
        assert value == pytest.approx(2 * 10 / 0.150)
        assert e2e == 75.0


def test_one_rank_needs_no_process_group():
    total, value = bench.replica_throughput(200.0, 10, 1, None, "cpu")
    assert total == 200.0 and value == pytest.approx(50.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun only rank 0 times the oracle and prints; other ranks exit
    without work (the workload dict is never touched)."""
    import argparse
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    bench.run_reference(args, None, rank=1)
    assert capsys.readouterr().out == ""
