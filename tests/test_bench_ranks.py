"""The benchmark's multi-rank host logic on CPU: gloo ranks in child processes (no GPU).

bench.py --gpus N runs N independent replicas of the layer (one per GPU, weak
scaling, no collective on the data path); the only cross-rank steps are the
barriers around the timed region and the max over ranks of the elapsed time.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], world)
        q.put((rank, ms, bench.whole_job_rate(4, world, ms, 100)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_rate(world):
    times = [10.0 + 7.5 * r for r in range(world)]  # the last rank is the slowest
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(times)
    for rank, ms, rate in got:
        assert ms == slowest
        # 4 tokens per rank per step, 100 steps, timed by the slowest rank
        assert rate == pytest.approx(4 * world * 100 / (slowest * 1e-3))


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_rate(4, 1, 32.0, 1000) == pytest.approx(4 * 1000 / 0.032)
