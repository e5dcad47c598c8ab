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


def _graph(seed, N=150, deg_max=9):
    """Receiver-sorted CSR of a random graph (senders anywhere, ascending per receiver)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    d = rng.integers(0, deg_max, N)
    d[rng.integers(0, N)] = 40   # one busier receiver
    rowptr = np.zeros(N + 1, np.int64)
    np.cumsum(d, out=rowptr[1:])
    sender = np.concatenate([np.sort(rng.integers(0, N, k)) for k in d]).astype(np.int64)
    return rowptr, sender


def test_halo_partition_local_graphs():
    """Each rank's local graph is its owned receivers' edges with senders renamed into the
    local index space (owned nodes, then the halo in ascending id); halo nodes have empty
    segments; the cuts cover the nodes and balance the edges to within one receiver."""
    import numpy as np
    from message_passing_gb300.halo import HaloPartition
    for seed in range(6):
        rowptr, sender = _graph(seed)
        N, E = rowptr.shape[0] - 1, int(rowptr[-1])
        dmax = int(np.diff(rowptr).max())
        for world in (1, 2, 3, 5):
            parts = [HaloPartition(rowptr, sender, world, r) for r in range(world)]
            assert parts[0].n0 == 0 and parts[-1].n1 == N
            for a, b in zip(parts[:-1], parts[1:]):
                assert a.n1 == b.n0 and a.e1 == b.e0
            for p in parts:
                assert abs((p.e1 - p.e0) - E / world) <= dmax
                assert p.rowptr.shape[0] == p.n_local + 1 and p.rowptr[-1] == p.e1 - p.e0
                assert np.all(p.rowptr[p.n_owned:] == p.e1 - p.e0)   # halo nodes receive nothing
                lut = np.concatenate([np.arange(p.n0, p.n1), p.halo])   # local id -> global id
                assert np.array_equal(lut[p.sender], sender[p.e0:p.e1])
                out = sender[p.e0:p.e1]
                out = out[(out < p.n0) | (out >= p.n1)]
                assert np.array_equal(p.halo, np.unique(out))
                assert np.array_equal(p.rowptr[:p.n_owned + 1], rowptr[p.n0:p.n1 + 1] - p.e0)


def _halo_worker(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from message_passing_gb300.halo import HaloPartition
    blocks, L, mul, scale = [(0, 1), (1, -1)], 2, 4, 0.3
    ot = oracle.table(blocks, L, L)
    rowptr, sender = _graph(21)
    N, E = rowptr.shape[0] - 1, int(rowptr[-1])
    rng = np.random.default_rng(4)
    x = rng.standard_normal((N, ot.d1, mul))
    y = oracle.sh(rng.standard_normal((E, 3)), L)
    w = rng.standard_normal((E, ot.n_paths, mul))
    dm = rng.standard_normal((N, ot.D, mul))
    p = HaloPartition(rowptr, sender, world, rank).setup()
    # forward: halo rows from their owners, then the local convolution (oracle as the compute)
    x_local = p.gather_halo(torch.from_numpy(x[p.n0:p.n1].copy())).numpy()
    yl, wl = y[p.e0:p.e1], w[p.e0:p.e1]
    m = oracle.conv_forward(ot, p.rowptr, p.sender, x_local, yl, wl, scale)[:p.n_owned]
    # backward: local dx partials (owned and halo senders) sent back to their owners
    dm_local = np.concatenate([dm[p.n0:p.n1], np.zeros((p.n_local - p.n_owned, ot.D, mul))])
    dx_local = oracle.conv_backward_dx(ot, p.rowptr, p.sender, yl, wl, dm_local, scale, Nq=mul)
    dx = p.scatter_halo_grad(torch.from_numpy(dx_local)).numpy()
    dy, dw = oracle.conv_backward_edges(ot, p.rowptr, p.sender, x_local, yl, wl, dm_local, scale)
    parts = [None] * world
    dist.all_gather_object(parts, (p.n0, m, dx, dy, dw))   # collected for the check only
    if rank == 0:
        parts.sort(key=lambda t: t[0])
        got = [np.concatenate([t[i] for t in parts]) for i in (1, 2, 3, 4)]
        want_m = oracle.conv_forward(ot, rowptr, sender, x, y, w, scale)
        want_dx = oracle.conv_backward_dx(ot, rowptr, sender, y, w, dm, scale, Nq=mul)
        want_dy, want_dw = oracle.conv_backward_edges(ot, rowptr, sender, x, y, w, dm, scale)
        ok = (np.array_equal(got[0], want_m) and np.array_equal(got[2], want_dy) and np.array_equal(got[3], want_dw)
              and np.allclose(got[1], want_dx, rtol=0, atol=1e-12 * np.abs(want_dx).max()))
        q.put(bool(ok))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_halo_conv_gloo(world):
    """One graph over gloo ranks: each convolves its receivers after the halo gather and
    returns the halo senders' dx partials to their owners. Messages, dy and dw equal the whole
    graph's bitwise; dx to rounding (its sums are split between ranks)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_halo_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    ok = q.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert ok


def test_halo_local_index():
    """local_index maps owned and halo nodes into the local index space, -1 elsewhere."""
    import numpy as np
    from message_passing_gb300.halo import HaloPartition
    rowptr, sender = _graph(5)
    N = rowptr.shape[0] - 1
    for world in (2, 4):
        for r in range(world):
            p = HaloPartition(rowptr, sender, world, r)
            lut = np.concatenate([np.arange(p.n0, p.n1), p.halo])
            li = p.local_index(np.arange(N))
            assert np.array_equal(np.nonzero(li >= 0)[0], np.sort(lut))
            assert np.array_equal(lut[li[li >= 0]], np.nonzero(li >= 0)[0])
            assert np.array_equal(p.local_index(lut), np.arange(p.n_local))
