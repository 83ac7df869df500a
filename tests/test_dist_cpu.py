"""The multi-rank host logic of bench.py on CPU: two gloo ranks (spawned
processes, 127.0.0.1) aggregate their step times the way the GPU run does
(the slowest rank's time, all ranks' boxes), and the reference arm does no
work on ranks other than 0.  No GPU is touched."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total, value = bench.aggregate_over_ranks(10.0 * (rank + 1), world, 8192, 5, device="cpu")
        out.put((rank, total, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, total, value in got:
        assert total == 20.0  # the slower rank's 20 ms
        assert value == pytest.approx(2 * 8192 * 5 / 0.020)


def test_single_rank_aggregation_needs_no_group():
    import bench
    assert bench.aggregate_over_ranks(8.0, 1, 1000, 4) == (8.0, 1000 * 4 / 0.008)


def test_reference_arm_idle_off_rank_zero(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="single_n8192", steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
