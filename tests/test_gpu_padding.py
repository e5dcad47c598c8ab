"""Padding edges on the GPU (e3j, Sec. 4 "Message passing convolution" and App. E: static-shape
graphs route unused edge slots to one padding node, and the kernels skip those edges).

A graph gets a padding node and padding edges (pad -> pad, pad -> real receivers, real
senders -> pad) whose inputs, and the padding node's rows, are NaN. With pad_node set, the
conv must (1) agree with the oracle's padding rule, (2) give every real output bit for bit
what the GPU gives on the graph without padding, and (3) write exact zeros to m[pad], dx[pad]
and the dy, dw rows of every padding edge (the output buffers start out NaN).
"""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
import synth
from gpu_util import TOL_BF16, TOL_F32, assert_close, sample_ids, to_dev, to_np
from synth import STREAM_GRAD, STREAM_W, device_normal
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()


def _nan_like_out(t, N, E, mul, dev):
    f = dict(dtype=torch.float32, device=dev)
    return (torch.full((N, t.D, mul), float("nan"), **f),
            (torch.full((N, t.d1, mul), float("nan"), **f), torch.full((E, t.d2), float("nan"), **f),
             torch.full((E, t.n_paths, mul), float("nan"), **f)))


def _run(t, g, xd, y, wd, dmd, scale, pad=-1):
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    m0, bw0 = _nan_like_out(t, g.n_nodes, g.n_edges, t.mul, xd.device)
    m = e3.conv_forward(t, rp, sd, xd, y, wd, scale, out=m0, pad_node=pad)
    csc = e3.graph_prepare(rp, sd, g.n_nodes)
    dx, dy, dw = e3.conv_backward(t, csc, xd, y, wd, dmd, scale, out=bw0, pad_node=pad)
    assert e3.check_device_status() == 0
    return m, dx, dy, dw


def _padded_inputs(g, gp, orig, xd, wd, dmd, dtype):
    """Device inputs of the padded graph: real rows copied from the unpadded ones, padding
    rows and the padding node's rows NaN."""
    dev = xd.device
    nan = float("nan")
    xp = torch.cat([xd, torch.full((1,) + tuple(xd.shape[1:]), nan, dtype=dtype, device=dev)])
    dmp = torch.cat([dmd, torch.full((1,) + tuple(dmd.shape[1:]), nan, dtype=dtype, device=dev)])
    wp = torch.full((gp.n_edges,) + tuple(wd.shape[1:]), nan, dtype=dtype, device=dev)
    real = np.nonzero(orig >= 0)[0]
    assert np.array_equal(orig[real], np.arange(g.n_edges))   # real edges keep their order
    for c in range(0, len(real), CH):
        wp[torch.from_numpy(real[c:c + CH]).to(dev)] = wd[c:c + CH]
    return xp, wp, dmp


CH = 1 << 18   # edge rows per chunk of the comparisons (bounded temporaries at full size)


def _rows_equal(a, ai, b):
    """a[ai] == b bit for bit (ai: numpy edge ids into a, in b's row order), in chunks."""
    for c in range(0, len(ai), CH):
        if not torch.equal(a[torch.from_numpy(ai[c:c + CH]).to(a.device)], b[c:c + CH]):
            return False
    return True


def _rows_zero(a, ai):
    for c in range(0, len(ai), CH):
        if not bool(torch.all(a[torch.from_numpy(ai[c:c + CH]).to(a.device)] == 0)):
            return False
    return True


def _check(blocks, mul, L2, L3, g, n_self, n_out, n_in, dtype, tol, k_nodes=None, k_edges=None, device_w=False):
    t = e3.Table.create(blocks, mul, L2, L3)
    ot = oracle.table(blocks, L2, L3)
    gp, pad, orig = synth.padded_graph(g, n_self, n_out, n_in, (97, g.n_edges))
    real = orig >= 0
    N, E = g.n_nodes, g.n_edges
    scale = N / max(E, 1)
    rng = np.random.default_rng(mul + E)
    xd = to_dev(rng.standard_normal((N, ot.d1, mul)).astype(np.float32), dtype)
    if device_w:
        wd = device_normal((E, ot.n_paths, mul), (96, STREAM_W), 1 / np.sqrt(ot.n_paths), dtype=dtype)
        dmd = device_normal((N, ot.D, mul), (96, STREAM_GRAD), dtype=dtype)
    else:
        wd = to_dev((rng.standard_normal((E, ot.n_paths, mul)) / np.sqrt(ot.n_paths)).astype(np.float32), dtype)
        dmd = to_dev(rng.standard_normal((N, ot.D, mul)).astype(np.float32), dtype)
    xp, wp, dmp = _padded_inputs(g, gp, orig, xd, wd, dmd, dtype)
    vec = g.vec.astype(np.float32)
    vecp = gp.vec.astype(np.float32)        # NaN on padding edges
    y = e3.sh_forward(to_dev(vec), L2, dtype=dtype)
    yp = e3.sh_forward(to_dev(vecp), L2, dtype=dtype)

    m, dx, dy, dw = _run(t, g, xd, y, wd, dmd, scale)
    mp, dxp, dyp, dwp = _run(t, gp, xp, yp, wp, dmp, scale, pad=pad)
    torch.cuda.synchronize()

    # (2) real outputs: bit for bit the unpadded graph's (real edge k of gp is edge k of g)
    dev = xd.device
    ridx, pidx = np.nonzero(real)[0], np.nonzero(~real)[0]
    assert torch.equal(mp[:N], m) and torch.equal(dxp[:N], dx)
    assert _rows_equal(dyp, ridx, dy) and _rows_equal(dwp, ridx, dw)
    # (3) exact zeros for the padding node and the padding edges
    assert torch.all(mp[pad] == 0) and torch.all(dxp[pad] == 0)
    assert _rows_zero(dyp, pidx) and _rows_zero(dwp, pidx)

    # (1) the oracle's padding rule on the padded graph (sampled rows at large sizes)
    xo, dmo = to_np(xp), to_np(dmp)
    yo = oracle.sh(vecp.astype(np.float64), L2)
    if dtype == torch.bfloat16:
        yo = to_np(torch.from_numpy(yo.astype(np.float32)).to(torch.bfloat16))
    wfetch = lambda ids: to_np(wp[torch.from_numpy(np.asarray(ids, np.int64)).to(dev)])
    Np, Ep = gp.n_nodes, gp.n_edges
    nodes = np.arange(Np) if k_nodes is None else np.union1d(sample_ids(Np, k_nodes, 21), [pad])
    edges = np.arange(Ep) if k_edges is None else np.union1d(sample_ids(Ep, k_edges, 22),
                                                             np.nonzero(~real)[0][:16])
    sel_n, sel_e = torch.from_numpy(nodes).to(dev), torch.from_numpy(edges).to(dev)
    ref_m = oracle.conv_forward(ot, gp.rowptr, gp.sender, xo, yo, wfetch, scale, receivers=nodes, pad_node=pad)
    assert_close(to_np(mp[sel_n]), ref_m, tol, "m")
    ref_dx = oracle.conv_backward_dx(ot, gp.rowptr, gp.sender, yo, wfetch, dmo, scale, senders=nodes, Nq=mul,
                                     pad_node=pad)
    assert_close(to_np(dxp[sel_n]), ref_dx, tol, "dx")
    ref_dy, ref_dw = oracle.conv_backward_edges(ot, gp.rowptr, gp.sender, xo, yo, wfetch, dmo, scale, edges=edges,
                                                pad_node=pad)
    assert_close(to_np(dyp[sel_e]), ref_dy, tol, "dy")
    assert_close(to_np(dwp[sel_e]), ref_dw, tol, "dw")


X2 = [(0, 1), (1, -1), (2, 1)]


@pytest.mark.parametrize("blocks,mul,L2,L3,dt", [
    (X2, 128, 3, 3, torch.float32),                            # 128-channel pipelined kernels
    (X2, 128, 3, 3, torch.bfloat16),
    ([(0, 1), (1, -1)], 128, 3, 3, torch.float32),
    ([(0, 1), (1, -1), (2, 1), (3, -1)], 8, 3, 3, torch.float32),   # plain kernels, 1 channel/lane
    ([(0, 1), (1, -1)], 64, 3, 3, torch.float32),              # plain kernels, 4 channels/lane
    ([(0, 1), (1, -1)], 16, 2, 2, torch.float32),
])
def test_padding_edges_skipped(blocks, mul, L2, L3, dt):
    g = synth.random_graph(300, 4000, (97, mul), empty_nodes=10)
    tol = TOL_BF16 if dt == torch.bfloat16 else TOL_F32
    # a third of the edges are padding, most of them on the padding node's own segment
    _check(blocks, mul, L2, L3, g, 1900, 60, 40, dt, tol)


def test_padding_only_graph():
    """Every edge is padding: all outputs are zero."""
    g = synth.random_graph(50, 0, (97, 1))
    _check(X2, 128, 3, 3, g, 700, 0, 0, torch.float32, TOL_F32)


def test_padding_full_size_64k_atoms():
    """The 64,000-atom workload's graph with a quarter of the edge slots padding (853k edges on
    one padding node, of 3.41 M), weights and gradients drawn on the device; sampled oracle rows,
    bitwise agreement with the unpadded graph everywhere."""
    w = W.WORKLOADS[4]
    g = W.make_graph(w)
    n_pad = g.n_edges // 3
    _check(X2, 128, 3, 3, g, n_pad - 60_000, 40_000, 20_000, torch.float32, TOL_F32, k_nodes=64, k_edges=256,
           device_w=True)
