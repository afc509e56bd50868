"""The benchmark's multi-rank logic on CPU: two gloo ranks, each with its own
timings, agree on the slowest rank's time and on the whole-job value."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 5.0 - rank, 0.0, 7.5 * (rank + 1)]
    got = bench.max_over_ranks(mine, dist, "cpu")
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = [10.0 + world - 1, 5.0, 0.0, 7.5 * world]
    for r in range(world):
        assert out[r] == want


def test_whole_job_value_is_replicas_over_slowest():
    # two replicas of 2e12 flops, the slower taking 2 ms: 2 * 2e12 / 2e-3 = 2000 TFLOP/s
    assert bench.whole_job_tflops(2e12, 2, 2.0) == pytest.approx(2000.0)
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([1.0, 2.0], None, "cpu") == [1.0, 2.0]
