"""The multi-rank host logic of bench.py (max-over-ranks timing, whole-job
throughput, barriers) on world_size-2 gloo process groups, CPU only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r ran slower steps: the job time is the slowest rank's
    steps = [1.0 + rank, 2.0 + rank, 3.0 + rank]
    total, per_step, value = bench.aggregate(steps, 64, world, "cpu")
    bench.barrier(world)
    out[rank] = (total, per_step, value, bench.reduce_max(float(rank * 10), world, "cpu"))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_aggregate_max_over_ranks(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    slow_total = sum([1.0 + world - 1, 2.0 + world - 1, 3.0 + world - 1])
    for r in range(world):
        total, per_step, value, mx = res[r]
        assert total == pytest.approx(slow_total)
        assert per_step == pytest.approx(slow_total / 3)
        assert value == pytest.approx(64 * world / (slow_total / 3 / 1e3))
        assert mx == (world - 1) * 10


def test_single_rank_aggregate():
    import bench
    total, per_step, value = bench.aggregate([2.0, 2.0], 100, 1, "cpu")
    assert total == 4.0 and per_step == 2.0 and value == pytest.approx(100 / 2e-3)
