"""Heavy real receivers: e3gb_conv_forward_split.

A receiver-stationary forward gives a receiver with very many edges to one warp (e3j, Sec. 4
"Message passing convolution": the receiver-degree imbalance deterministic kernels face). The
split forward cuts such a segment into pieces summed by separate warps and added in piece order.
Checked against the float64 oracle on a graph with one real hub receiver of 100,000 edges,
bitwise against e3gb_conv_forward on every receiver at or under the chunk, for bitwise
repeatability, and for time (the unsplit forward sums the hub on one warp).
"""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
from gpu_util import TOL_BF16, TOL_F32, assert_close, to_dev, to_np
from synth import Graph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()


def _hub_graph(n_nodes, hub_deg, deg, seed):
    """Receiver-sorted CSR: node 17 receives hub_deg edges, every other node deg (random
    senders, unit-free random edge vectors)."""
    rng = np.random.default_rng(seed)
    d = np.full(n_nodes, deg, np.int64)
    d[17] = hub_deg
    rowptr = np.zeros(n_nodes + 1, np.int64)
    np.cumsum(d, out=rowptr[1:])
    E = int(rowptr[-1])
    sender = rng.integers(0, n_nodes, E)
    for b in range(n_nodes):   # senders ascending within a receiver, as the workloads have them
        sender[rowptr[b]:rowptr[b + 1]].sort()
    vec = rng.standard_normal((E, 3))
    return Graph(n_nodes, rowptr.astype(np.int32), sender.astype(np.int32), vec, 0.0, 0.0, "hub")


@pytest.mark.parametrize("blocks,mul", [([(0, 1), (1, -1)], 128),                 # pipelined forward
                                        ([(0, 1), (1, -1), (2, 1), (3, -1)], 8)])  # edge-slot forward
def test_split_forward_heavy_receiver(blocks, mul):
    L = 3
    t = e3.Table.create(blocks, mul, L, L)
    ot = oracle.table(blocks, L, L)
    g = _hub_graph(600, 100_000, 30, 5)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((g.n_nodes, ot.d1, mul)).astype(np.float32)
    w = (rng.standard_normal((g.n_edges, ot.n_paths, mul)) / np.sqrt(ot.n_paths)).astype(np.float32)
    scale = g.n_nodes / g.n_edges
    rp, sd, xd, wd = to_dev(g.rowptr), to_dev(g.sender), to_dev(x), to_dev(w)
    v32 = g.vec.astype(np.float32)
    y = e3.sh_forward(to_dev(v32), L)
    chunk = 1024
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record()
    ms = e3.conv_forward_split(t, rp, sd, xd, y, wd, scale, chunk=chunk)
    ev[1].record()
    m1 = e3.conv_forward(t, rp, sd, xd, y, wd, scale)
    ev[2].record()
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    # receivers at or under the chunk: exactly the unsplit result
    light = np.nonzero(np.diff(g.rowptr) <= chunk)[0]
    li = torch.from_numpy(light).cuda()
    assert torch.equal(ms[li], m1[li])
    # the hub and a few others against the oracle
    yo = oracle.sh(v32.astype(np.float64), L)
    rcv = np.array([0, 16, 17, 18, 599])
    ref = oracle.conv_forward(ot, g.rowptr, g.sender, x, yo, w, scale, receivers=rcv)
    got = to_np(ms[torch.from_numpy(rcv).cuda()])
    # each against the RMS of its own rows: the hub's sums of 100,000 edges are ~60x the
    # others' (30 edges), so one RMS over both would not be the scale of either
    assert_close(got[[0, 1, 3, 4]], ref[[0, 1, 3, 4]], TOL_F32, "m (neighbours)")
    assert_close(got[2], ref[2], TOL_F32, "m (hub)")
    # bitwise repeatable
    for _ in range(3):
        assert torch.equal(ms, e3.conv_forward_split(t, rp, sd, xd, y, wd, scale, chunk=chunk))
    # the split forward does not wait for one warp to sum 100k edges
    t_split, t_plain = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
    assert t_split < 0.5 * t_plain, (t_split, t_plain)


def test_split_forward_padding_and_small_chunks():
    """A padding node with a heavy segment is still passed over whole; chunk = 1 (every edge a
    piece) and chunk larger than every degree give the oracle's result."""
    blocks, mul, L = [(0, 1), (1, -1)], 16, 2
    t = e3.Table.create(blocks, mul, L, L)
    ot = oracle.table(blocks, L, L)
    g = _hub_graph(120, 3000, 12, 7)
    pad = 17   # the hub is the padding node here: its segment must be skipped, m[pad] = 0
    rng = np.random.default_rng(8)
    x = rng.standard_normal((g.n_nodes, ot.d1, mul)).astype(np.float32)
    w = (rng.standard_normal((g.n_edges, ot.n_paths, mul)) / np.sqrt(ot.n_paths)).astype(np.float32)
    v32 = g.vec.astype(np.float32)
    yo = oracle.sh(v32.astype(np.float64), L)
    y = e3.sh_forward(to_dev(v32), L)
    ref = oracle.conv_forward(ot, g.rowptr, g.sender, x, yo, w, 0.3, pad_node=pad)
    for chunk in (1, 5, 64, 100_000):
        m = e3.conv_forward_split(t, to_dev(g.rowptr), to_dev(g.sender), to_dev(x), y, to_dev(w), 0.3, chunk=chunk,
                                  pad_node=pad)
        torch.cuda.synchronize()
        assert e3.check_device_status() == 0
        assert torch.all(m[pad] == 0)
        assert_close(to_np(m), ref, TOL_F32, f"m (chunk {chunk})")


@pytest.mark.parametrize("blocks", [[(0, 1), (1, -1)],              # plain bf16 forward
                                    [(0, 1), (1, -1), (2, 1)]])     # pipelined bf16 forward
def test_split_forward_heavy_receiver_bf16(blocks):
    """bf16 storage, fp32 sums: a hub of 20,000 edges against the oracle on the same stored
    bf16 inputs (harmonics included), and bitwise equal to the unsplit forward elsewhere."""
    mul, L = 128, 3
    t = e3.Table.create(blocks, mul, L, L)
    ot = oracle.table(blocks, L, L)
    g = _hub_graph(300, 20_000, 24, 9)
    rng = np.random.default_rng(10)
    bf = torch.bfloat16
    xd = to_dev(rng.standard_normal((g.n_nodes, ot.d1, mul)).astype(np.float32), bf)
    wd = to_dev((rng.standard_normal((g.n_edges, ot.n_paths, mul)) / np.sqrt(ot.n_paths)).astype(np.float32), bf)
    v32 = g.vec.astype(np.float32)
    yb = torch.from_numpy(oracle.sh(v32.astype(np.float64), L).astype(np.float32)).to(bf)
    yd = yb.cuda()
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    scale = g.n_nodes / g.n_edges
    ms = e3.conv_forward_split(t, rp, sd, xd, yd, wd, scale, chunk=512)
    m1 = e3.conv_forward(t, rp, sd, xd, yd, wd, scale)
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    light = torch.from_numpy(np.nonzero(np.diff(g.rowptr) <= 512)[0]).cuda()
    assert torch.equal(ms[light], m1[light])
    rcv = np.array([0, 17, 299])
    ref = oracle.conv_forward(ot, g.rowptr, g.sender, to_np(xd), to_np(yb), to_np(wd), scale, receivers=rcv)
    got = to_np(ms[torch.from_numpy(rcv).cuda()])
    assert_close(got[1], ref[1], TOL_BF16, "m (hub)")
    assert_close(got[[0, 2]], ref[[0, 2]], TOL_BF16, "m (neighbours)")
