"""The N>1 host logic of bench.py on CPU: two gloo ranks, one process each.

Each rank times its own replica; the job's time is the slowest rank's and its
rows are the sum over ranks. The data path has no collective, so the only
cross-rank traffic is the barrier and these two scalar reductions.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist("gloo")
    try:
        d.barrier()
        ms = d.max(10.0 + rank)              # rank 1 is the slower one
        rows = d.sum(8192.0 * (rank + 1))
        q.put((rank, d.world, ms, rows))
    finally:
        d.close()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, world, ms, rows in got:
        assert world == 2
        assert ms == 11.0
        assert rows == 8192.0 * 3


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist("gloo")
    assert d.dist is None and d.max(3.0) == 3.0 and d.sum(4.0) == 4.0


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
