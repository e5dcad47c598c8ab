"""Edge cases, index validation on the device, the sender-major index and determinism."""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
from gpu_util import TOL_F32, assert_close, to_dev, to_np
from synth import random_graph
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()   # start from a clean error word
    yield
    torch.cuda.synchronize()


def _setup(blocks, mul, N, E, seed, empty=0, L2=3, L3=3):
    t = e3.Table.create(blocks, mul, L2, L3)
    ot = oracle.table(blocks, L2, L3)
    g = random_graph(N, E, (95, seed), empty_nodes=empty)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, ot.d1, mul)).astype(np.float32)
    w = (rng.standard_normal((E, ot.n_paths, mul)) / np.sqrt(ot.n_paths)).astype(np.float32)
    dm = rng.standard_normal((N, ot.D, mul)).astype(np.float32)
    return t, ot, g, x, w, dm


def test_graph_prepare_matches_stable_sort():
    g = random_graph(700, 9000, (95, 1), empty_nodes=50)
    # a few heavy senders and receivers
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    cp, ce, cr = e3.graph_prepare(rp, sd, g.n_nodes)
    assert e3.check_device_status() == 0
    order = np.argsort(g.sender, kind="stable")
    ptr = np.zeros(g.n_nodes + 1, np.int64)
    np.cumsum(np.bincount(g.sender, minlength=g.n_nodes), out=ptr[1:])
    assert np.array_equal(cp.cpu().numpy(), ptr)
    assert np.array_equal(ce.cpu().numpy(), order)
    assert np.array_equal(cr.cpu().numpy(), g.receiver()[order])


def test_graph_prepare_heavy_sender_and_receiver():
    N = 300
    recv = np.concatenate([np.zeros(2500, np.int64), np.arange(1, N)])
    send = np.concatenate([np.random.default_rng(2).integers(0, N, 2500), np.full(N - 1, 7)])
    srt = np.lexsort((send, recv))
    recv, send = recv[srt], send[srt]
    rowptr = np.zeros(N + 1, np.int64)
    np.cumsum(np.bincount(recv, minlength=N), out=rowptr[1:])
    cp, ce, cr = e3.graph_prepare(to_dev(rowptr.astype(np.int32)), to_dev(send.astype(np.int32)), N)
    assert e3.check_device_status() == 0
    order = np.argsort(send, kind="stable")
    assert np.array_equal(ce.cpu().numpy(), order)
    assert np.array_equal(cr.cpu().numpy(), recv[order])


def test_graph_prepare_padding_node_of_huge_valency():
    """Static-shape graphs send their unused edge slots from one padding node (e3j, Sec. 4
    "Message passing convolution"): here 600k of 1M edges. The index must still be numpy's
    stable argsort bit for bit, and its cost linear in the edges: well under 50 ms."""
    N = 20_001
    pad = N - 1
    rng = np.random.default_rng(7)
    n_real, n_pad_in, n_pad = 380_000, 20_000, 600_000
    recv = np.concatenate([rng.integers(0, pad, n_real), rng.integers(0, pad, n_pad_in), np.full(n_pad, pad)])
    send = np.concatenate([rng.integers(0, pad, n_real), np.full(n_pad_in, pad), np.full(n_pad, pad)])
    srt = np.argsort(recv, kind="stable")
    recv, send = recv[srt], send[srt]
    rowptr = np.zeros(N + 1, np.int64)
    np.cumsum(np.bincount(recv, minlength=N), out=rowptr[1:])
    rp, sd = to_dev(rowptr.astype(np.int32)), to_dev(send.astype(np.int32))
    cp, ce, cr = e3.graph_prepare(rp, sd, N)
    ws = torch.empty(e3.graph_prepare_workspace_bytes(N, len(send)), dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    e3.graph_prepare(rp, sd, N, out=(cp, ce, cr), workspace=ws)
    ev[1].record()
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    order = np.argsort(send, kind="stable")
    ptr = np.zeros(N + 1, np.int64)
    np.cumsum(np.bincount(send, minlength=N), out=ptr[1:])
    assert np.array_equal(cp.cpu().numpy(), ptr)
    assert np.array_equal(ce.cpu().numpy(), order)
    assert np.array_equal(cr.cpu().numpy(), recv[order])
    assert ev[0].elapsed_time(ev[1]) < 50.0


def test_graph_prepare_edges_outside_rowptr_left_out():
    """Edges before rowptr[0] or from rowptr[N] on belong to no receiver: they are left out
    of the index (not flagged), and the entries past csc_ptr[N] are -1."""
    g = random_graph(50, 600, (95, 3))
    rp = g.rowptr.copy()
    lo, hi = int(rp[1]), int(rp[-2])
    rp[0], rp[-1] = lo, hi           # receiver 0 and receiver N-1 lose their edges
    cp, ce, cr = e3.graph_prepare(to_dev(rp), to_dev(g.sender), g.n_nodes)
    assert e3.check_device_status() == 0
    keep = np.arange(lo, hi)
    order = keep[np.argsort(g.sender[keep], kind="stable")]
    n = len(keep)
    assert int(cp[-1]) == n
    assert np.array_equal(ce.cpu().numpy()[:n], order)
    assert np.all(ce.cpu().numpy()[n:] == -1) and np.all(cr.cpu().numpy()[n:] == -1)
    assert np.array_equal(cr.cpu().numpy()[:n], g.receiver()[order])


def _run(t, g, x, w, dm, scale):
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    y = e3.sh_forward(to_dev(g.vec.astype(np.float32)), t.sh_lmax)
    xd, wd, dmd = to_dev(x), to_dev(w), to_dev(dm)
    m = e3.conv_forward(t, rp, sd, xd, y, wd, scale)
    csc = e3.graph_prepare(rp, sd, g.n_nodes)
    dx, dy, dw = e3.conv_backward(t, csc, xd, y, wd, dmd, scale)
    return m, dx, dy, dw


def test_empty_graph():
    t, ot, g, x, w, dm = _setup([(0, 1), (1, -1)], 32, 6, 0, 3)
    rp = to_dev(g.rowptr)
    sd = torch.zeros(0, dtype=torch.int32, device="cuda")
    xd = to_dev(x)
    m = torch.full((6, t.D, 32), 7.0, device="cuda")
    e3.conv_forward(t, rp, sd, xd, torch.zeros((0, 16), device="cuda"),
                    torch.zeros((0, t.n_paths, 32), device="cuda"), 1.0, out=m)
    assert torch.all(m == 0)
    csc = e3.graph_prepare(rp, sd, 6)
    dx = torch.full_like(xd, 7.0)
    e3.conv_backward(t, csc, xd, torch.zeros((0, 16), device="cuda"), torch.zeros((0, t.n_paths, 32), device="cuda"),
                     to_dev(dm), 1.0, out=(dx, torch.zeros((0, 16), device="cuda"),
                                           torch.zeros((0, t.n_paths, 32), device="cuda")))
    assert torch.all(dx == 0)
    assert e3.check_device_status() == 0


@pytest.mark.parametrize("mul", [4, 8, 64])
def test_star_graph_and_isolated_nodes(mul):
    """One receiver with every edge; every other node only sends."""
    t = e3.Table.create([(0, 1), (1, -1)], mul, 3, 3)
    ot = oracle.table([(0, 1), (1, -1)], 3, 3)
    N = 97
    rowptr = np.zeros(N + 1, np.int32)
    rowptr[1:] = N - 1
    sender = np.arange(1, N, dtype=np.int32)
    rng = np.random.default_rng(4)
    vec = rng.standard_normal((N - 1, 3)).astype(np.float32)
    x = rng.standard_normal((N, ot.d1, mul)).astype(np.float32)
    w = rng.standard_normal((N - 1, ot.n_paths, mul)).astype(np.float32)
    dm = rng.standard_normal((N, ot.D, mul)).astype(np.float32)
    from synth import Graph
    g = Graph(N, rowptr, sender, vec.astype(np.float64))
    m, dx, dy, dw = _run(t, g, x, w, dm, 0.5)
    y = oracle.sh(vec.astype(np.float64), 3)
    ref_m = oracle.conv_forward(ot, rowptr, sender, x, y, w, 0.5)
    # only receiver 0 has edges: its own RMS sets the scale; the rest must be exactly zero
    assert_close(to_np(m)[:1], ref_m[:1], TOL_F32, "m")
    assert np.all(to_np(m)[1:] == 0.0)
    assert_close(to_np(dx), oracle.conv_backward_dx(ot, rowptr, sender, y, w, dm, 0.5), TOL_F32, "dx")
    rdy, rdw = oracle.conv_backward_edges(ot, rowptr, sender, x, y, w, dm, 0.5)
    assert_close(to_np(dy), rdy, TOL_F32, "dy")
    assert_close(to_np(dw), rdw, TOL_F32, "dw")


def test_determinism_bitwise():
    w = W.WORKLOADS[3]
    t = e3.Table.create(w.blocks, w.mul, 3, 3)
    g = W.make_graph(w, n_atoms=1500)
    P = t.n_paths
    x, ww = W.make_conv(w, g, P)
    dm = W.make_grad(w, g.n_nodes, t.D)
    first = [o.clone() for o in _run(t, g, x, ww, dm, 0.02)]
    for _ in range(9):
        again = _run(t, g, x, ww, dm, 0.02)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    # bf16 storage at 128 channels (the plain forward on this configuration)
    xb, wb, dmb = (torch.from_numpy(a).to(torch.bfloat16) for a in (x, ww, dm))
    yb = e3.sh_forward(to_dev(g.vec.astype(np.float32)), 3, dtype=torch.bfloat16)
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    xb, wb = xb.cuda(), wb.cuda()
    m0 = e3.conv_forward(t, rp, sd, xb, yb, wb, 0.02)
    for _ in range(9):
        assert torch.equal(m0, e3.conv_forward(t, rp, sd, xb, yb, wb, 0.02))
    # 8 channels: the edge-slot forward, whose slot sums are added in a fixed order
    w5 = W.WORKLOADS[5]
    t5 = e3.Table.create(w5.blocks, w5.mul, 3, 3)
    g5 = W.make_graph(w5, n_atoms=1500)
    x5, ww5 = W.make_conv(w5, g5, t5.n_paths)
    dm5 = W.make_grad(w5, g5.n_nodes, t5.D)
    first = [o.clone() for o in _run(t5, g5, x5, ww5, dm5, 0.03)]
    for _ in range(9):
        for a, b in zip(first, _run(t5, g5, x5, ww5, dm5, 0.03)):
            assert torch.equal(a, b)
    # rows: TP forward / backward
    w2 = W.WORKLOADS[2]
    t2 = e3.Table.create(w2.blocks, w2.mul, 3, 3)
    u, x2, w2w = W.make_tp(w2, t2.n_paths, rows=999)
    y = e3.sh_forward(to_dev(u.astype(np.float32)), 3)
    xd, wd = to_dev(x2), to_dev(w2w)
    dz = torch.randn((999, t2.D, 128), device="cuda")
    z0 = e3.tp_forward(t2, xd, y, wd)
    b0 = [o.clone() for o in e3.tp_backward(t2, xd, y, wd, dz)]
    for _ in range(9):
        assert torch.equal(z0, e3.tp_forward(t2, xd, y, wd))
        for a, b in zip(b0, e3.tp_backward(t2, xd, y, wd, dz)):
            assert torch.equal(a, b)


def test_out_of_range_sender_is_skipped_and_flagged():
    t, ot, g, x, w, dm = _setup([(0, 1), (1, -1)], 16, 40, 300, 5)
    bad = g.sender.copy()
    bad[17] = 40 + 3          # sender outside [0, N)
    bad[200] = -1
    rp, sd = to_dev(g.rowptr), to_dev(bad)
    y = e3.sh_forward(to_dev(g.vec.astype(np.float32)), 3)
    m = e3.conv_forward(t, rp, sd, to_dev(x), y, to_dev(w), 1.0)
    with pytest.raises(e3.E3GBError) as ex:
        e3.check_device_status()
    assert ex.value.status == e3.ERR_DEVICE_INDEX
    # the result equals the oracle on the graph without those two edges (weights zeroed)
    w0 = w.copy()
    w0[[17, 200]] = 0.0
    yo = oracle.sh(g.vec.astype(np.float32).astype(np.float64), 3)
    assert_close(to_np(m), oracle.conv_forward(ot, g.rowptr, g.sender, x, yo, w0, 1.0), TOL_F32, "m")
    # the sender-major index leaves the two edges out and flags them
    cp, ce, cr = e3.graph_prepare(rp, sd, 40)
    with pytest.raises(e3.E3GBError):
        e3.check_device_status()
    assert int(cp[-1]) == 298
    assert e3.check_device_status() == 0     # cleared


def test_bad_rowptr_is_flagged():
    t, ot, g, x, w, dm = _setup([(0, 1), (1, -1)], 16, 20, 100, 6)
    rp = g.rowptr.copy()
    assert rp[5] >= 3
    rp[6] = rp[5] - 3                                       # a decreasing pointer
    rp[7] = 10 ** 6                                         # beyond n_edges
    y = e3.sh_forward(to_dev(g.vec.astype(np.float32)), 3)
    e3.conv_forward(t, to_dev(rp), to_dev(g.sender), to_dev(x), y, to_dev(w), 1.0)
    with pytest.raises(e3.E3GBError) as ex:
        e3.check_device_status()
    assert ex.value.status == e3.ERR_DEVICE_INDEX
    e3.graph_prepare(to_dev(rp), to_dev(g.sender), 20)
    with pytest.raises(e3.E3GBError):
        e3.check_device_status()


def test_host_pointer_rejected():
    t = e3.Table.create([(0, 1), (1, -1)], 16, 2, 2)
    xh = torch.zeros((4, t.d1, 16))
    yd = torch.zeros((4, t.d2), device="cuda")
    wd = torch.zeros((4, t.n_paths, 16), device="cuda")
    zd = torch.zeros((4, t.D, 16), device="cuda")
    with pytest.raises(e3.E3GBError) as ex:
        e3.tp_forward(t, xh, yd, wd, out=zd)
    assert ex.value.status == e3.ERR_INVALID_ARG
