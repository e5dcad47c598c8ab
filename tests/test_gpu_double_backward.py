"""Convolution double backward on the GPU (e3j App. E.1 Eq. (17)-(18)) against the oracle's
composition of first-order conv / conv_bwd calls, plus padding, determinism and agreement
with the same composition run on the GPU's own first-order kernels."""
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

X2 = [(0, 1), (1, -1), (2, 1)]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()


def _inputs(ot, N, E, mul, dtype, seed, device_w=False):
    r = np.random.default_rng(seed)
    dev = lambda a: to_dev(a.astype(np.float32), dtype)
    d = dict(x=dev(r.standard_normal((N, ot.d1, mul))), dm=dev(r.standard_normal((N, ot.D, mul))),
             ddx=dev(r.standard_normal((N, ot.d1, mul))), ddy=dev(r.standard_normal((E, ot.d2))))
    if device_w:
        d["w"] = device_normal((E, ot.n_paths, mul), (98, STREAM_W), 1 / np.sqrt(ot.n_paths), dtype=dtype)
        d["ddw"] = device_normal((E, ot.n_paths, mul), (98, STREAM_GRAD), 1 / np.sqrt(ot.n_paths), dtype=dtype)
    else:
        d["w"] = dev(r.standard_normal((E, ot.n_paths, mul)) / np.sqrt(ot.n_paths))
        d["ddw"] = dev(r.standard_normal((E, ot.n_paths, mul)) / np.sqrt(ot.n_paths))
    return d


def _gpu(t, g, d, y, scale, pad=-1):
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    csc = e3.graph_prepare(rp, sd, g.n_nodes)
    out = e3.conv_double_backward(t, rp, sd, csc, d["x"], y, d["w"], d["dm"], d["ddx"], d["ddy"], d["ddw"], scale,
                                  pad_node=pad)
    assert e3.check_device_status() == 0
    return out


def _oracle(ot, g, d, vec32, L2, dtype, scale, nodes=None, edges=None, pad=None):
    yo = oracle.sh(vec32.astype(np.float64), L2)
    if dtype == torch.bfloat16:
        yo = to_np(torch.from_numpy(yo.astype(np.float32)).to(torch.bfloat16))
    fetch = lambda t: (lambda ids: to_np(t[torch.from_numpy(np.asarray(ids, np.int64)).cuda()]))
    return oracle.conv_double_backward(ot, g.rowptr, g.sender, to_np(d["x"]), yo, fetch(d["w"]), to_np(d["dm"]),
                                       to_np(d["ddx"]), fetch(d["ddy"]), fetch(d["ddw"]), scale, receivers=nodes,
                                       senders=nodes, edges=edges, pad_node=pad)


def _compare(out, ref, tol, nodes=None, edges=None):
    gx, gy, gw, gdm = out
    sel_n = slice(None) if nodes is None else torch.from_numpy(nodes).cuda()
    sel_e = slice(None) if edges is None else torch.from_numpy(edges).cuda()
    assert_close(to_np(gx[sel_n]), ref[0], tol, "delta_x")
    assert_close(to_np(gy[sel_e]), ref[1], tol, "delta_y")
    assert_close(to_np(gw[sel_e]), ref[2], tol, "delta_w")
    assert_close(to_np(gdm[sel_n]), ref[3], tol, "delta_dm")


@pytest.mark.parametrize("blocks,mul,L2,L3,dt", [
    (X2, 128, 3, 3, torch.float32),
    (X2, 128, 3, 3, torch.bfloat16),
    ([(0, 1), (1, -1), (2, 1), (3, -1)], 8, 3, 3, torch.float32),
    ([(0, 1), (1, -1)], 64, 3, 3, torch.float32),
    ([(0, 1), (1, -1)], 16, 2, 2, torch.float32),
    ([(1, -1)], 32, 1, 2, torch.float32),                       # one output block per path
])
def test_double_backward_matches_oracle(blocks, mul, L2, L3, dt):
    per_path = blocks == [(1, -1)]
    t = e3.Table.create(blocks, mul, L2, L3, per_path=per_path)
    ot = oracle.table(blocks, L2, L3, per_path=per_path)
    g = synth.random_graph(260, 3000, (98, mul), empty_nodes=7)
    scale = g.n_nodes / g.n_edges
    d = _inputs(ot, g.n_nodes, g.n_edges, mul, dt, mul)
    vec32 = g.vec.astype(np.float32)
    y = e3.sh_forward(to_dev(vec32), L2, dtype=dt)
    out = _gpu(t, g, d, y, scale)
    torch.cuda.synchronize()
    _compare(out, _oracle(ot, g, d, vec32, L2, dt, scale), TOL_BF16 if dt == torch.bfloat16 else TOL_F32)


def test_double_backward_equals_gpu_composition_and_is_deterministic():
    """The fused passes equal Eq. (17)-(18) composed from the GPU's own conv and conv_bwd
    (within fp32 summation-order differences) and repeat bit for bit."""
    t = e3.Table.create(X2, 128, 3, 3)
    ot = oracle.table(X2, 3, 3)
    g = W.make_graph(W.WORKLOADS[4], n_atoms=600)
    scale = g.n_nodes / g.n_edges
    d = _inputs(ot, g.n_nodes, g.n_edges, 128, torch.float32, 5)
    y = e3.sh_forward(to_dev(g.vec.astype(np.float32)), 3)
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    csc = e3.graph_prepare(rp, sd, g.n_nodes)
    a = _gpu(t, g, d, y, scale)
    b = _gpu(t, g, d, y, scale)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    x, w, dm, ddx, ddy, ddw = (d[k] for k in ("x", "w", "dm", "ddx", "ddy", "ddw"))
    ddm = (e3.conv_forward(t, rp, sd, ddx, y, w, scale) + e3.conv_forward(t, rp, sd, x, ddy, w, scale)
           + e3.conv_forward(t, rp, sd, x, y, ddw, scale))
    _, dy1, dw1 = e3.conv_backward(t, csc, ddx, y, w, dm, scale)
    dx2, _, dw2 = e3.conv_backward(t, csc, x, ddy, w, dm, scale)
    dx3, dy3, _ = e3.conv_backward(t, csc, x, y, ddw, dm, scale)
    torch.cuda.synchronize()
    # both sides are fp32 results each within TOL_F32 x RMS of the exact one, so they may
    # differ by twice that
    for got, ref, name in ((a[0], dx2 + dx3, "delta_x"), (a[1], dy1 + dy3, "delta_y"), (a[2], dw1 + dw2, "delta_w"),
                           (a[3], ddm, "delta_dm")):
        assert_close(to_np(got), to_np(ref), 2 * TOL_F32, name)


def test_double_backward_padding():
    t = e3.Table.create(X2, 128, 3, 3)
    ot = oracle.table(X2, 3, 3)
    g = synth.random_graph(200, 2500, (98, 1))
    gp, pad, orig = synth.padded_graph(g, 1000, 40, 30, (98, 2))
    real = orig >= 0
    scale = 0.25
    d = _inputs(ot, g.n_nodes, g.n_edges, 128, torch.float32, 9)
    nan = float("nan")

    def node_pad(v):
        return torch.cat([v, torch.full((1,) + tuple(v.shape[1:]), nan, device=v.device)])

    def edge_pad(v):
        o = torch.full((gp.n_edges,) + tuple(v.shape[1:]), nan, device=v.device)
        o[torch.from_numpy(np.nonzero(real)[0]).cuda()] = v
        return o
    dp = {k: (node_pad(v) if k in ("x", "dm", "ddx") else edge_pad(v)) for k, v in d.items()}
    y = e3.sh_forward(to_dev(g.vec.astype(np.float32)), 3)
    yp = e3.sh_forward(to_dev(gp.vec.astype(np.float32)), 3)
    a = _gpu(t, g, d, y, scale)
    b = _gpu(t, gp, dp, yp, scale, pad=pad)
    torch.cuda.synchronize()
    ridx = torch.from_numpy(np.nonzero(real)[0]).cuda()
    pidx = torch.from_numpy(np.nonzero(~real)[0]).cuda()
    N = g.n_nodes
    assert torch.equal(b[0][:N], a[0]) and torch.equal(b[3][:N], a[3])
    assert torch.equal(b[1][ridx], a[1]) and torch.equal(b[2][ridx], a[2])
    assert torch.all(b[0][pad] == 0) and torch.all(b[3][pad] == 0)
    assert torch.all(b[1][pidx] == 0) and torch.all(b[2][pidx] == 0)
    _compare(b, _oracle(ot, gp, dp, gp.vec.astype(np.float32), 3, torch.float32, scale, pad=pad), TOL_F32)


def test_double_backward_full_size_sampled():
    """The 64,000-atom / 2.56 M-edge workload, weights and their variations drawn on the
    device; sampled nodes and edges against the oracle."""
    wl = W.WORKLOADS[4]
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    ot = oracle.table(wl.blocks, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl)
    scale = g.n_nodes / g.n_edges
    d = _inputs(ot, g.n_nodes, g.n_edges, wl.mul, torch.float32, 4, device_w=True)
    vec32 = g.vec.astype(np.float32)
    y = e3.sh_forward(to_dev(vec32), 3)
    out = _gpu(t, g, d, y, scale)
    torch.cuda.synchronize()
    nodes, edges = sample_ids(g.n_nodes, 48, 31), sample_ids(g.n_edges, 192, 32)
    _compare(out, _oracle(ot, g, d, vec32, 3, torch.float32, scale, nodes, edges), TOL_F32, nodes, edges)
