"""The bench's multi-rank host logic on two CPU ranks (gloo): every rank gets the slowest
rank's time, the job value counts the units of all ranks over that time, and the
reference arm prints nothing on ranks other than 0.  No GPU: the data path of a rank is
an independent replica, so only this aggregation crosses ranks."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [40.0, 55.0][rank]
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_throughput(world, 1000, 10, ms)
        q.put((rank, ms, value, bench.rank_info()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value, info in got:
        assert ms == 55.0                                  # the slowest rank's time everywhere
        assert value == pytest.approx(2 * 1000 * 10 / 0.055)
        assert info == (rank, 2, 0)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(None, bench.WORKLOADS["layer-T32"]) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(1, 100, 4, 2.0) == pytest.approx(200000.0)
