"""The multi-rank logic of bench.py on CPU (gloo, two ranks, no GPU).

Every rank runs its own replica of the workload (weak scaling, no data-path
collective); the job is timed by its slowest rank.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(times[rank])
    value = bench.whole_job_tflops(world, 10**12, slowest)
    out.put((rank, slowest, value, bench.dist_env()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [2.0, 5.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, env in results:
        assert slowest == 5.0
        # two replicas of 1 TFLOP each in 5 ms
        assert value == pytest.approx(2 * 10**12 / 5e-3 / 1e12)
        assert env == (rank, world, rank)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 2 * 10**12, 4.0) == pytest.approx(500.0)
