"""The receiver-range partition of one graph (message_passing_gb300.halo) on the GPU: every
rank's local graph (its receivers, the halo senders renamed, empty segments for the halo
nodes) goes through the library's convolution kernels on one GPU, rank after rank, with the
halo exchanges done by indexing. Messages, dy and dw of the assembled result equal the whole
graph's bitwise (same rows, same per-receiver order); dx, whose sums are split between ranks,
to the fp32 tolerance. The exchanges themselves are covered by the gloo tests."""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
from gpu_util import TOL_F32, assert_close, to_np
from message_passing_gb300.halo import HaloPartition
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("world", [2, 3])
def test_partitioned_conv_matches_whole_graph(world):
    w = W.WORKLOADS[3]   # 128x(0e+1o), SH l<=3, rc 5 A
    t = e3.Table.create(w.blocks, w.mul, w.sh_lmax, w.out_lmax)
    g = W.make_graph(w, n_atoms=600)
    N, E = g.n_nodes, g.n_edges
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((N, t.d1, w.mul)).astype(np.float32)).cuda()
    wd = torch.from_numpy((rng.standard_normal((E, t.n_paths, w.mul)) / 4).astype(np.float32)).cuda()
    dm = torch.from_numpy(rng.standard_normal((N, t.D, w.mul)).astype(np.float32)).cuda()
    y = e3.sh_forward(torch.from_numpy(g.vec.astype(np.float32)).cuda(), w.sh_lmax)
    scale = N / E
    rp, sd = torch.from_numpy(g.rowptr).cuda(), torch.from_numpy(g.sender).cuda()
    m_whole = e3.conv_forward(t, rp, sd, x, y, wd, scale)
    dx_whole, dy_whole, dw_whole = e3.conv_backward(t, e3.graph_prepare(rp, sd, N), x, y, wd, dm, scale)
    parts = [HaloPartition(g.rowptr, g.sender, world, r) for r in range(world)]
    m, dy, dw, dx_part = [], [], [], []
    for p in parts:
        lut = torch.from_numpy(np.concatenate([np.arange(p.n0, p.n1), p.halo])).cuda()
        x_local = x[lut].contiguous()                                   # the forward halo gather
        lrp, lsd = torch.from_numpy(p.rowptr).cuda(), torch.from_numpy(p.sender).cuda()
        yl, wl = y[p.e0:p.e1], wd[p.e0:p.e1]
        m.append(e3.conv_forward(t, lrp, lsd, x_local, yl, wl, scale)[:p.n_owned])
        dm_local = torch.zeros((p.n_local, t.D, w.mul), device="cuda")
        dm_local[:p.n_owned] = dm[p.n0:p.n1]
        gx, gy, gw = e3.conv_backward(t, e3.graph_prepare(lrp, lsd, p.n_local), x_local, yl, wl, dm_local, scale)
        dy.append(gy)
        dw.append(gw)
        dx_part.append(gx)
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    assert torch.equal(torch.cat(m), m_whole)
    assert torch.equal(torch.cat(dy), dy_whole)
    assert torch.equal(torch.cat(dw), dw_whole)
    # the backward halo exchange: owners add the peers' partials in ascending rank
    dx = torch.cat([gx[:p.n_owned] for p, gx in zip(parts, dx_part)])
    for r, p in enumerate(parts):
        halo = torch.from_numpy(p.halo).cuda()
        if halo.numel():
            dx[halo] += dx_part[r][p.n_owned:]
    assert_close(to_np(dx), to_np(dx_whole), TOL_F32, "dx")


def test_partitioned_conv_with_padding_node():
    """A padded graph (one padding node, 20% padding edge slots, NaN in its rows and the
    padding edges' inputs) over 3 ranks: each passes the padding node's local id (owned or
    halo, -1 if absent) as pad_node. Real outputs equal the whole padded graph's."""
    import synth
    w = W.WORKLOADS[3]
    t = e3.Table.create(w.blocks, w.mul, w.sh_lmax, w.out_lmax)
    g0 = W.make_graph(w, n_atoms=500)
    n_pad = g0.n_edges // 4
    g, pad, orig = synth.padded_graph(g0, n_pad - n_pad // 10, n_pad // 20, n_pad // 20, (w.wid, 9))
    N, E = g.n_nodes, g.n_edges
    rng = np.random.default_rng(8)
    x = torch.from_numpy(rng.standard_normal((N, t.d1, w.mul)).astype(np.float32)).cuda()
    x[pad] = float("nan")
    wd = torch.from_numpy((rng.standard_normal((E, t.n_paths, w.mul)) / 4).astype(np.float32)).cuda()
    wd[torch.from_numpy(np.nonzero(orig < 0)[0]).cuda()] = float("nan")
    dm = torch.from_numpy(rng.standard_normal((N, t.D, w.mul)).astype(np.float32)).cuda()
    dm[pad] = float("nan")
    vec = g.vec.astype(np.float32).copy()
    vec[orig < 0] = 1.0   # the harmonics of padding slots are never read either
    y = e3.sh_forward(torch.from_numpy(vec).cuda(), w.sh_lmax)
    scale = N / E
    rp, sd = torch.from_numpy(g.rowptr).cuda(), torch.from_numpy(g.sender).cuda()
    m_whole = e3.conv_forward(t, rp, sd, x, y, wd, scale, pad_node=pad)
    dx_whole, dy_whole, dw_whole = e3.conv_backward(t, e3.graph_prepare(rp, sd, N), x, y, wd, dm, scale,
                                                    pad_node=pad)
    parts = [HaloPartition(g.rowptr, g.sender, 3, r) for r in range(3)]
    m, dy, dw, dx_part = [], [], [], []
    for p in parts:
        lpad = int(p.local_index([pad])[0])
        lut = torch.from_numpy(np.concatenate([np.arange(p.n0, p.n1), p.halo])).cuda()
        x_local = x[lut].contiguous()
        lrp, lsd = torch.from_numpy(p.rowptr).cuda(), torch.from_numpy(p.sender).cuda()
        yl, wl = y[p.e0:p.e1], wd[p.e0:p.e1]
        m.append(e3.conv_forward(t, lrp, lsd, x_local, yl, wl, scale, pad_node=lpad)[:p.n_owned])
        dm_local = torch.zeros((p.n_local, t.D, w.mul), device="cuda")
        dm_local[:p.n_owned] = dm[p.n0:p.n1]
        gx, gy, gw = e3.conv_backward(t, e3.graph_prepare(lrp, lsd, p.n_local), x_local, yl, wl, dm_local, scale,
                                      pad_node=lpad)
        dy.append(gy)
        dw.append(gw)
        dx_part.append(gx)
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    assert torch.equal(torch.cat(m), m_whole)
    assert torch.equal(torch.cat(dy), dy_whole)
    assert torch.equal(torch.cat(dw), dw_whole)
    dx = torch.cat([gx[:p.n_owned] for p, gx in zip(parts, dx_part)])
    for r, p in enumerate(parts):
        halo = torch.from_numpy(p.halo).cuda()
        if halo.numel():
            dx[halo] += dx_part[r][p.n_owned:]
    real = torch.from_numpy(np.setdiff1d(np.arange(N), [pad])).cuda()
    assert bool(torch.isfinite(dx[real]).all())
    assert torch.all(dx[pad] == 0) and torch.all(dx_whole[pad] == 0)
    assert_close(to_np(dx[real]), to_np(dx_whole[real]), TOL_F32, "dx")
