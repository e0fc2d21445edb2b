"""The multi-GPU form of the bench is replicas only (one draft step is a serial
chain; nothing in it shards): each rank times its own steps, the ranks agree on
the slowest rank's time with an all-reduce MAX, and the whole-job rate counts
every rank's steps.  Checked here with two gloo ranks on the CPU."""
from __future__ import annotations

import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import torch.distributed as d
    import bench
    d.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        mine = [12.5, 20.0, 7.0][rank]
        slowest = bench.barrier_max(ws, mine, device="cpu")
        q.put((rank, slowest, bench.whole_job_rate(10, ws, slowest)))
    finally:
        d.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 3])
def test_ranks_agree_on_the_slowest_time_and_count_every_rank(ws):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = max([12.5, 20.0, 7.0][:ws])
    for rank, slowest, rate in got:
        assert slowest == want
        assert rate == pytest.approx(10 * ws / (want / 1000))


def test_single_rank_is_its_own_time():
    import bench
    assert bench.barrier_max(1, 3.5) == 3.5
    assert bench.whole_job_rate(20, 1, 10.0) == pytest.approx(2000.0)
