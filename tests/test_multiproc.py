"""The multi-rank host logic of the bench on CPU: two gloo ranks, each timing its own replica of the step;
the job's time is the slowest rank's and the value aggregates the bytes of every rank (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, "cpu")
        q.put((rank, ms, bench.aggregate_rate(1000, 4, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]                 # max over ranks on both
    assert res[0][2] == pytest.approx(1000 * 4 * 2 / 0.015 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
