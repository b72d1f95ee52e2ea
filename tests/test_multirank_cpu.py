"""The multi-process path of bench.py on CPU: two gloo ranks, 127.0.0.1.

Each rank is a replica (the conv shards with no exchange), so the only
cross-rank steps are the barrier around the timed region and the
max-over-ranks of its duration; the whole-job value is the bytes all ranks
moved divided by the slowest rank's time.  The reference arm runs on rank 0
alone; other ranks exit without work.
"""

from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist = bench.Dist(world, "gloo")
    dist.barrier()
    region_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    ms_per_step, value = bench.aggregate(dist, world, 1_000_000, region_ms, 5, "cpu")
    dist.barrier()
    dist.close()
    out.put((rank, ms_per_step, value))


def test_two_rank_aggregation_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms_per_step, value in res:
        assert ms_per_step == pytest.approx(20.0 / 5)  # the slowest rank's 20 ms over 5 steps
        assert value == pytest.approx(2 * 1_000_000 / 4e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert capsys.readouterr().out == ""
