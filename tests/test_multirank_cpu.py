"""The N > 1 paths on CPU with the gloo backend: bench.py's aggregation (independent
replicas, one per rank: every rank reports the slowest rank's time and the whole-job rate
counts the units of all ranks), and the data-parallel split of a batch of independent
graphs (shard_graphs), whose ranks compute on their own graphs with no exchange."""
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


def _batch(seed, n_graphs=7, d1=4, mul=8, n_paths=None):
    """A batch of small random graphs stored as one CSR (edges stay inside their graph)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    sizes = rng.integers(1, 12, n_graphs)
    gp = np.concatenate([[0], np.cumsum(sizes)])
    rowptr, sender = [0], []
    for g in range(n_graphs):
        for b in range(gp[g], gp[g + 1]):
            deg = int(rng.integers(0, 6))
            sender += sorted(int(v) for v in rng.integers(gp[g], gp[g + 1], deg))
            rowptr.append(rowptr[-1] + deg)
    return gp, np.array(rowptr, np.int64), np.array(sender, np.int64)


def test_shard_graphs_partition():
    """Shards are contiguous, cover every node and edge once, never cut a graph, keep every
    edge's sender inside the shard, and split the edges evenly up to one graph's edges."""
    import numpy as np
    import message_passing_gb300 as e3
    for seed in range(20):
        gp, rp, sd = _batch(seed, n_graphs=int(3 + seed % 9))
        E = int(rp[-1])
        big = int(np.max(rp[gp[1:]] - rp[gp[:-1]]))
        for world in (1, 2, 3, 5):
            parts = [e3.shard_graphs(gp, rp, sd, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[0][2] == 0
            assert parts[-1][1] == gp[-1] and parts[-1][3] == E
            for r in range(world - 1):
                assert parts[r][1] == parts[r + 1][0] and parts[r][3] == parts[r + 1][2]
            for n0, n1, e0, e1 in parts:
                assert n0 in gp and n1 in gp                       # whole graphs
                assert np.all((sd[e0:e1] >= n0) & (sd[e0:e1] < n1))  # no edge leaves the shard
                assert e0 == rp[n0] and e1 == rp[n1]
                assert abs((e1 - e0) - E / world) <= big + 1


def test_shard_graphs_rejects_cross_edges():
    import numpy as np
    import message_passing_gb300 as e3
    gp, rp, sd = _batch(3)
    sd = sd.copy()
    sd[0] = gp[-1] - 1   # an edge into graph 0 from the last graph
    with pytest.raises(ValueError):
        e3.shard_graphs(gp, rp, sd, 2, 0)


def _conv_worker(rank, world, port, q):
    import numpy as np
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import message_passing_gb300 as e3
    import oracle
    blocks, L = [(0, 1), (1, -1)], 2
    ot = oracle.table(blocks, L, L)
    gp, rp, sd = _batch(11, n_graphs=9)
    rng = np.random.default_rng(5)
    N, E, mul = int(gp[-1]), int(rp[-1]), 8
    x = rng.standard_normal((N, ot.d1, mul))
    vec = rng.standard_normal((E, 3))
    w = rng.standard_normal((E, ot.n_paths, mul))
    y = oracle.sh(vec, L)
    n0, n1, e0, e1 = e3.shard_graphs(gp, rp, sd, world, rank)
    # this rank's own graphs only: its CSR, its nodes' x, its edges' y and w
    m = oracle.conv_forward(ot, rp[n0:n1 + 1] - e0, sd[e0:e1] - n0, x[n0:n1], y[e0:e1], w[e0:e1], 0.5)
    parts = [None] * world
    dist.all_gather_object(parts, (n0, m))   # collected for the check only
    if rank == 0:
        whole = oracle.conv_forward(ot, rp, sd, x, y, w, 0.5)
        got = np.concatenate([p[1] for p in sorted(parts, key=lambda p: p[0])])
        q.put(bool(np.array_equal(got, whole)) and got.shape == whole.shape)
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_conv_gloo():
    """Two gloo ranks each run the (oracle) convolution on their shard of a batch of graphs;
    the shards' outputs, concatenated, are bitwise the convolution of the whole batch."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_conv_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=180)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert ok
