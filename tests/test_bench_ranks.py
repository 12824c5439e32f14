"""The multi-rank logic of bench.py on the CPU: two gloo ranks, each with its own time; both
must see the slowest rank's time, and the whole-job rate counts every rank's tokens.  Under
torchrun the reference arm runs on rank 0 only (other ranks return without work)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 95.5][rank]
        m = bench.reduce_max(local_ms, "cpu")
        rate = bench.throughput(4096, 10, world, m)
        q.put((rank, m, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, rate in got:
        assert m == 120.0
        assert rate == pytest.approx(4096 * 10 * 2 / 0.120)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    ns = type("A", (), dict(workload="tiny_f32", steps=1, warmup=0, gpus=2, cpu_seconds=1.0))()
    assert bench.run_reference(ns) is None
    assert capsys.readouterr().out == ""
