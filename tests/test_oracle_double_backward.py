"""Pins of the oracle's convolution double backward (oracle.conv_double_backward, e3j App. E.1
Eq. (17)-(18)).

The double backward is the gradient of L(x, y, w, dm) = <dx, ddx> + <dy, ddy> + <dw, ddw>,
where (dx, dy, dw) is the first-order backward (itself pinned by finite differences of the
forward). The backward is linear in each of x, y, w, dm with the others held fixed, so L is
affine along any one of them and a finite difference with step 1 is exact up to rounding:
<delta_x, v> = L(x + v) - L(x), and so on for y, w and dm. None of this uses Eq. (17)-(18).
"""
import numpy as np
import pytest

import oracle
import synth


def _case(blocks, Nq, seed, L2=3, L3=3, N=25, E=140):
    t = oracle.table(blocks, L2, L3)
    g = synth.random_graph(N, E, (79, seed), empty_nodes=2)
    r = np.random.default_rng(seed)
    arrs = dict(x=r.standard_normal((N, t.d1, Nq)), y=r.standard_normal((E, t.d2)),
                w=r.standard_normal((E, t.n_paths, Nq)), dm=r.standard_normal((N, t.D, Nq)),
                ddx=r.standard_normal((N, t.d1, Nq)), ddy=r.standard_normal((E, t.d2)),
                ddw=r.standard_normal((E, t.n_paths, Nq)))
    return t, g, arrs, r


def _L(t, g, a, scale):
    dy, dw = oracle.conv_backward_edges(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"], scale)
    dx = oracle.conv_backward_dx(t, g.rowptr, g.sender, a["y"], a["w"], a["dm"], scale, Nq=a["x"].shape[2])
    return (dx * a["ddx"]).sum() + (dy * a["ddy"]).sum() + (dw * a["ddw"]).sum()


@pytest.mark.parametrize("blocks,Nq,L2,L3", [([(0, 1), (1, -1)], 3, 3, 3), ([(0, 1), (1, -1), (2, 1)], 2, 3, 3),
                                             ([(1, -1)], 4, 1, 2)])
def test_double_backward_is_gradient_of_pairing(blocks, Nq, L2, L3):
    t, g, a, r = _case(blocks, Nq, 3 + Nq, L2, L3)
    scale = 0.7
    gx, gy, gw, gdm = oracle.conv_double_backward(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"],
                                                  a["ddx"], a["ddy"], a["ddw"], scale)
    L0 = _L(t, g, a, scale)
    for name, grad in (("x", gx), ("y", gy), ("w", gw), ("dm", gdm)):
        v = r.standard_normal(a[name].shape)
        moved = dict(a)
        moved[name] = a[name] + v
        exact = _L(t, g, moved, scale) - L0
        assert abs((grad * v).sum() - exact) <= 1e-10 * max(1.0, abs(exact)), name


def test_double_backward_euler_identities():
    """L is linear in dm and affine in x, y, w: <delta_dm, dm> = L; <delta_x, x> = <dy, ddy> +
    <dw, ddw>; <delta_y, y> = <dx, ddx> + <dw, ddw>; <delta_w, w> = <dx, ddx> + <dy, ddy>."""
    t, g, a, _ = _case([(0, 1), (1, -1)], 4, 11)
    gx, gy, gw, gdm = oracle.conv_double_backward(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"],
                                                  a["ddx"], a["ddy"], a["ddw"], 1.3)
    dy, dw = oracle.conv_backward_edges(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"], 1.3)
    dx = oracle.conv_backward_dx(t, g.rowptr, g.sender, a["y"], a["w"], a["dm"], 1.3, Nq=4)
    px, py, pw = (dx * a["ddx"]).sum(), (dy * a["ddy"]).sum(), (dw * a["ddw"]).sum()
    np.testing.assert_allclose((gdm * a["dm"]).sum(), px + py + pw, rtol=1e-12)
    np.testing.assert_allclose((gx * a["x"]).sum(), py + pw, rtol=1e-12)
    np.testing.assert_allclose((gy * a["y"]).sum(), px + pw, rtol=1e-12)
    np.testing.assert_allclose((gw * a["w"]).sum(), px + py, rtol=1e-12)


def test_double_backward_subsets_and_padding():
    """Sampled receivers / senders / edges equal the full result's rows; with a padding node
    the real rows equal the unpadded graph's."""
    t, g, a, _ = _case([(0, 1), (1, -1)], 3, 12)
    full = oracle.conv_double_backward(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"], a["ddx"], a["ddy"],
                                       a["ddw"], 0.5)
    nodes, edges = np.array([0, 3, 7, 24]), np.array([1, 5, 80, 139])
    sub = oracle.conv_double_backward(t, g.rowptr, g.sender, a["x"], a["y"], a["w"], a["dm"], a["ddx"], a["ddy"],
                                      a["ddw"], 0.5, receivers=nodes, senders=nodes, edges=edges)
    np.testing.assert_array_equal(sub[0], full[0][nodes])
    np.testing.assert_array_equal(sub[1], full[1][edges])
    np.testing.assert_array_equal(sub[2], full[2][edges])
    np.testing.assert_array_equal(sub[3], full[3][nodes])
    gp, pad, orig = synth.padded_graph(g, 30, 5, 5, (79, 99))
    real = orig >= 0

    def node_pad(v):
        return np.concatenate([v, np.full((1,) + v.shape[1:], np.nan)])

    def edge_pad(v):
        o = np.full((gp.n_edges,) + v.shape[1:], np.nan)
        o[real] = v[orig[real]]
        return o
    padded = oracle.conv_double_backward(t, gp.rowptr, gp.sender, node_pad(a["x"]), edge_pad(a["y"]),
                                         edge_pad(a["w"]), node_pad(a["dm"]), node_pad(a["ddx"]), edge_pad(a["ddy"]),
                                         edge_pad(a["ddw"]), 0.5, pad_node=pad)
    np.testing.assert_array_equal(padded[0][:-1], full[0])
    np.testing.assert_array_equal(padded[3][:-1], full[3])
    np.testing.assert_array_equal(padded[1][real], full[1][orig[real]])
    np.testing.assert_array_equal(padded[2][real], full[2][orig[real]])
    assert np.all(padded[1][~real] == 0) and np.all(padded[2][~real] == 0)
    assert np.all(padded[0][pad] == 0) and np.all(padded[3][pad] == 0)
