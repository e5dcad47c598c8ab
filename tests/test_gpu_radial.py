"""Parity of the radial edge-scalar path with the float64 oracle.

The radial convolution forms each edge's weights w[e] = h[e] @ W2 inside the kernels, from
the hidden activations h = silu(bessel_basis(|r_e|) @ W1) (e3j, App. E.1 notation for the edge
scalars s; App. A.3 "Linear mixing"). The oracle computes the same quantities as the plain
composition: oracle.radial.weights, then its convolution on those weights, then
hidden_from_weights_cotangent for dh. Tolerances: the hidden layer (a per-edge function)
max |err| <= 1e-5 RMS(oracle); the convolution outputs and forces, whose radial weights are
heavy-tailed, max |err| <= 1.5e-6 max|oracle| (the fp32 bound of the drawn-weight workloads
relative to the maximum; see gpu_util).
"""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
from gpu_util import TOL_F32, TOL_F32_MAX, assert_close, assert_close_max, sample_ids, to_dev, to_np
from oracle import radial
from synth import random_graph
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_radial_hidden_and_its_backward():
    rc = 4.571
    rng = np.random.default_rng(11)
    n = 3001
    vec = rng.standard_normal((n, 3))
    vec *= (rng.uniform(0.0, 1.25 * rc, n) / np.linalg.norm(vec, axis=1))[:, None]
    vec[0] = 0.0                        # the d -> 0 limit, no gradient
    vec[1] = (rc, 0.0, 0.0)             # at the cutoff: h = 0
    vec[2] = (0.0, 0.0, 1.3 * rc)       # beyond it
    v32 = vec.astype(np.float32)
    W1 = (2.0 * rng.standard_normal((8, 8))).astype(np.float32)
    h = e3.radial_hidden(to_dev(v32), to_dev(W1), rc)
    vo = v32.astype(np.float64)
    rc32 = float(np.float32(rc))        # the library takes r_cut as fp32
    assert_close(to_np(h), radial.hidden(vo, W1, rc32), TOL_F32, "h")
    assert np.all(to_np(h)[1:3] == 0.0)
    dh = rng.standard_normal((n, 8)).astype(np.float32)
    dvec = e3.radial_backward(to_dev(v32), to_dev(W1), rc, to_dev(dh))
    ref = radial.hidden_backward(vo, W1, rc32, dh)
    assert_close(to_np(dvec), ref, TOL_F32, "dvec")   # one float64 evaluation per edge, rounded once
    assert np.all(to_np(dvec)[0] == 0.0)
    # accumulate adds to what is there
    base = torch.ones((n, 3), device="cuda")
    e3.radial_backward(to_dev(v32), to_dev(W1), rc, to_dev(dh), out=base, accumulate=True)
    assert_close(to_np(base), ref + 1.0, TOL_F32, "dvec accumulated")
    # other basis and hidden sizes (the hidden kernel takes any up to 16)
    W1b = rng.standard_normal((5, 12)).astype(np.float32)
    hb = e3.radial_hidden(to_dev(v32), to_dev(W1b), 3.0)
    assert_close(to_np(hb), radial.hidden(vo, W1b, 3.0), TOL_F32, "h (5 basis, 12 hidden)")


def _radial_case(wl, g, ot, mul=None):
    mul = wl.mul if mul is None else mul
    rng = np.random.default_rng(wl.wid + 50)
    x = rng.standard_normal((g.n_nodes, ot.d1, mul)).astype(np.float32)
    dm = rng.standard_normal((g.n_nodes, ot.D, mul)).astype(np.float32)
    W1 = (2.0 * rng.standard_normal((8, 8))).astype(np.float32)
    W2 = (rng.standard_normal((8, ot.n_paths, mul)) / np.sqrt(8 * ot.n_paths)).astype(np.float32)
    return x, dm, W1, W2


def _gpu_radial(t, g, x, dm, W1, W2, rc, scale, pad=-1):
    v = to_dev(g.vec.astype(np.float32))
    rp, sd = to_dev(g.rowptr), to_dev(g.sender)
    y = e3.sh_forward(v, t.sh_lmax)
    h = e3.radial_hidden(v, to_dev(W1), rc)
    W2d = to_dev(W2)
    xd, dmd = to_dev(x), to_dev(dm)
    m = e3.conv_forward_radial(t, rp, sd, xd, y, h, W2d, scale, pad_node=pad)
    csc = e3.graph_prepare(rp, sd, g.n_nodes)
    dx, dy, dh = e3.conv_backward_radial(t, csc, xd, y, h, W2d, dmd, scale, pad_node=pad)
    # forces: through the harmonics plus through the radial weights
    dvec = e3.sh_backward(v, dy, t.sh_lmax)
    e3.radial_backward(v, to_dev(W1), rc, dh, out=dvec, accumulate=True)
    torch.cuda.synchronize()
    return m, dx, dy, dh, dvec


# (workload, atoms, channels): 128 channels run the pipelined kernels, others the plain ones
CASES = [(3, 400, None), (4, 500, None), (5, 1500, None), (4, 300, 64), (3, 300, 16)]


@pytest.mark.parametrize("wid,atoms,mul", CASES)
def test_conv_radial_matches_oracle(wid, atoms, mul):
    wl = W.WORKLOADS[wid]
    mul = wl.mul if mul is None else mul
    t = e3.Table.create(wl.blocks, mul, wl.sh_lmax, wl.out_lmax)
    ot = oracle.table(wl.blocks, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=atoms)
    rc = float(g.cutoff)
    x, dm, W1, W2 = _radial_case(wl, g, ot, mul)
    scale = g.n_nodes / g.n_edges
    m, dx, dy, dh, dvec = _gpu_radial(t, g, x, dm, W1, W2, rc, scale)
    assert e3.check_device_status() == 0
    vo = g.vec.astype(np.float32).astype(np.float64)
    yo = oracle.sh(vo, wl.sh_lmax)
    rc32 = float(np.float32(rc))
    wo = radial.weights(vo, W1, W2, rc32)
    assert_close_max(to_np(m), oracle.conv_forward(ot, g.rowptr, g.sender, x, yo, wo, scale), TOL_F32_MAX, "m")
    assert_close_max(to_np(dx), oracle.conv_backward_dx(ot, g.rowptr, g.sender, yo, wo, dm, scale), TOL_F32_MAX,
                     "dx")
    rdy, rdw = oracle.conv_backward_edges(ot, g.rowptr, g.sender, x, yo, wo, dm, scale)
    assert_close_max(to_np(dy), rdy, TOL_F32_MAX, "dy")
    rdh = radial.hidden_from_weights_cotangent(rdw, W2)
    assert_close_max(to_np(dh), rdh, TOL_F32_MAX, "dh")
    rf = oracle.sh_grad(vo, wl.sh_lmax, rdy) + radial.hidden_backward(vo, W1, rc32, rdh)
    assert_close_max(to_np(dvec), rf, TOL_F32_MAX, "forces")


def test_conv_radial_deterministic():
    wl = W.WORKLOADS[4]
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    ot = oracle.table(wl.blocks, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=400)
    x, dm, W1, W2 = _radial_case(wl, g, ot)
    first = _gpu_radial(t, g, x, dm, W1, W2, float(g.cutoff), 0.5)
    for _ in range(4):
        again = _gpu_radial(t, g, x, dm, W1, W2, float(g.cutoff), 0.5)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("wid,atoms", [(4, 400), (5, 600)])
def test_conv_radial_padding(wid, atoms):
    """Padding edges (one padding node, NaN in every padding input) leave the real outputs
    bitwise equal to the unpadded graph's; the padding rows of dy and dh are zero."""
    import synth
    wl = W.WORKLOADS[wid]
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    ot = oracle.table(wl.blocks, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=atoms)
    x, dm, W1, W2 = _radial_case(wl, g, ot)
    rc, scale = float(g.cutoff), 0.25
    m0, dx0, dy0, dh0, _ = _gpu_radial(t, g, x, dm, W1, W2, rc, scale)
    n_pad = g.n_edges // 3
    gp, pad, orig = synth.padded_graph(g, n_pad - 40, 25, 15, (wl.wid, 19))
    gp.vec[orig < 0] = np.nan
    xp = np.concatenate([x, np.full((1,) + x.shape[1:], np.nan, np.float32)])
    dmp = np.concatenate([dm, np.full((1,) + dm.shape[1:], np.nan, np.float32)])
    v = to_dev(gp.vec.astype(np.float32))
    rp, sd = to_dev(gp.rowptr), to_dev(gp.sender)
    y = e3.sh_forward(v, t.sh_lmax)
    h = e3.radial_hidden(v, to_dev(W1), rc)
    m = e3.conv_forward_radial(t, rp, sd, to_dev(xp), y, h, to_dev(W2), scale, pad_node=pad)
    csc = e3.graph_prepare(rp, sd, gp.n_nodes)
    dx, dy, dh = e3.conv_backward_radial(t, csc, to_dev(xp), y, h, to_dev(W2), to_dev(dmp), scale, pad_node=pad)
    torch.cuda.synchronize()
    assert e3.check_device_status() == 0
    real = orig >= 0
    assert torch.equal(m[:pad], m0) and torch.all(m[pad] == 0)
    assert torch.equal(dx[:pad], dx0) and torch.all(dx[pad] == 0)
    ri = torch.from_numpy(np.nonzero(real)[0]).cuda()
    pi = torch.from_numpy(np.nonzero(~real)[0]).cuda()
    assert torch.equal(dy[ri], dy0[torch.from_numpy(orig[real]).cuda()])
    assert torch.equal(dh[ri], dh0[torch.from_numpy(orig[real]).cuda()])
    assert torch.all(dy[pi] == 0) and torch.all(dh[pi] == 0)


def test_conv_radial_full_size_sampled():
    """The 64,000-atom workload (2.56 M edges) in the launch configuration the benchmark
    times: sampled receivers, senders and edges against the oracle, computed one by one."""
    wl = W.WORKLOADS[4]
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    ot = oracle.table(wl.blocks, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl)
    x, dm, W1, W2 = _radial_case(wl, g, ot)
    rc, scale = float(g.cutoff), g.n_nodes / g.n_edges
    m, dx, dy, dh, _ = _gpu_radial(t, g, x, dm, W1, W2, rc, scale)
    assert e3.check_device_status() == 0
    vo = g.vec.astype(np.float32).astype(np.float64)
    yf = lambda ids: oracle.sh(vo[ids], wl.sh_lmax)
    wf = lambda ids: radial.weights(vo[ids], W1, W2, float(np.float32(rc)))
    rcv = sample_ids(g.n_nodes, 48, 1)
    assert_close_max(to_np(m[torch.from_numpy(rcv).cuda()]),
                     oracle.conv_forward(ot, g.rowptr, g.sender, x, yf, wf, scale, receivers=rcv), TOL_F32_MAX, "m")
    snd = sample_ids(g.n_nodes, 48, 2)
    assert_close_max(to_np(dx[torch.from_numpy(snd).cuda()]),
                     oracle.conv_backward_dx(ot, g.rowptr, g.sender, yf, wf, dm, scale, senders=snd), TOL_F32_MAX,
                     "dx")
    eds = sample_ids(g.n_edges, 256, 3)
    rdy, rdw = oracle.conv_backward_edges(ot, g.rowptr, g.sender, x, yf, wf, dm, scale, edges=eds)
    ei = torch.from_numpy(eds).cuda()
    assert_close_max(to_np(dy[ei]), rdy, TOL_F32_MAX, "dy")
    assert_close_max(to_np(dh[ei]), radial.hidden_from_weights_cotangent(rdw, W2), TOL_F32_MAX, "dh")


def test_conv_radial_rejects_unsupported():
    wl = W.WORKLOADS[3]
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    g = random_graph(10, 30, (95, 9))
    x = torch.zeros((10, t.d1, t.mul), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((30, t.d2), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((30, 8), device="cuda")
    W2 = torch.zeros((8, t.n_paths, t.mul), device="cuda")
    with pytest.raises(e3.E3GBError) as ex:
        e3.conv_forward_radial(t, to_dev(g.rowptr), to_dev(g.sender), x, y, h, W2, 1.0)
    assert ex.value.status == e3.ERR_UNSUPPORTED
