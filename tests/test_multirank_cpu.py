"""The N > 1 aggregation of bench.py (independent replicas, one per rank) with the gloo
backend on CPU: every rank reports the slowest rank's time and the whole-job rate counts the
units of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.0 + rank, device="cpu")      # rank r took 1 + r seconds
    q.put((rank, t, bench.whole_job_rate(1000, 5, world, t)))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, t, rate in out:
        assert t == float(world)                      # slowest rank: 1 + (world - 1)
        assert rate == 1000 * 5 * world / float(world)


def test_single_process_is_local_time():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.whole_job_rate(10, 4, 1, 2.0) == 20.0
