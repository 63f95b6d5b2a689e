"""The multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.  Each rank
runs its own workload (weak scaling, no collective on the data path); the bench only
synchronises the ranks around the timed region and takes the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    slowest = bench.max_over_ranks(world, 1.0 + rank)   # rank 1 is the slower one
    value = bench.job_throughput(100.0, slowest, world)
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, slowest, value))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.0, 2.0]
    assert [o[2] for o in out] == [100.0, 100.0]   # 2 ranks x 100 units / 2 s


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1, 3.5) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0
