"""Pins of the oracle's tensor product and convolution (oracle/tp.c via oracle/__init__.py).

"e3j ...", App. E.1: Eq. (10)-(11) tensor product weighted per path and channel,
Eq. (12)-(13) message-passing convolution, Eq. (14)-(16) backward rules; App. A.1 Eq. (1)-(3)
equivariance.
"""
import math

import numpy as np
import pytest
from scipy.spatial.transform import Rotation

import oracle
from oracle.sh import sh, sh_l
from synth import random_graph

BLOCKS4 = [(0, 1), (1, -1), (2, 1)]
BLOCKS5 = [(0, 1), (1, -1), (2, 1), (3, -1)]


def _units(n, seed):
    g = np.random.default_rng(seed).standard_normal((n, 3))
    return g / np.linalg.norm(g, axis=1, keepdims=True)


def _wigner(R, l):
    u = _units(200, 21)
    return np.linalg.lstsq(sh_l(u, l), sh_l(u @ R.T, l), rcond=None)[0].T


def _rotate_x(t, x, R):
    xr = x.copy()
    off = 0
    for l, _ in t.blocks:
        D = _wigner(R, l)
        xr[:, off:off + 2 * l + 1, :] = np.einsum("ij,rjq->riq", D, x[:, off:off + 2 * l + 1, :])
        off += 2 * l + 1
    return xr


def _rotate_z(t, z, R):
    zr = z.copy()
    off = 0
    for l, _ in t.out_blocks:
        D = _wigner(R, l)
        zr[:, off:off + 2 * l + 1, :] = np.einsum("ij,rjq->riq", D, z[:, off:off + 2 * l + 1, :])
        off += 2 * l + 1
    return zr


def _parity_x(t, x):
    s = np.concatenate([np.full(2 * l + 1, p, float) for l, p in t.blocks])
    return x * s[None, :, None]


def _parity_z(t, z):
    s = np.concatenate([np.full(2 * l + 1, p, float) for l, p in t.out_blocks])
    return z * s[None, :, None]


def _inputs(t, R, Nq, seed):
    g = np.random.default_rng(seed)
    u = _units(R, seed + 1) * g.uniform(0.5, 2.0, (R, 1))
    return u, g.standard_normal((R, t.d1, Nq)), g.standard_normal((R, t.n_paths, Nq))


@pytest.mark.parametrize("blocks,per_path", [(BLOCKS4, False), (BLOCKS5, False), (BLOCKS4, True)])
def test_tp_equivariance_rotation_and_parity(blocks, per_path):
    t = oracle.table(blocks, 3, 3, per_path)
    u, x, w = _inputs(t, 6, 5, 1)
    z = oracle.tp_forward(t, x, sh(u, 3), w)
    R = Rotation.random(random_state=3).as_matrix()
    zr = oracle.tp_forward(t, _rotate_x(t, x, R), sh(u @ R.T, 3), w)
    np.testing.assert_allclose(zr, _rotate_z(t, z, R), atol=1e-11)
    zp = oracle.tp_forward(t, _parity_x(t, x), sh(-u, 3), w)
    np.testing.assert_allclose(zp, _parity_z(t, z), atol=1e-12)


def test_tp_closed_forms_l1():
    """x = 1o, SH l <= 1, one output block per path: identity, dot and cross products."""
    t = oracle.table([(1, -1)], 1, 2, per_path=True)
    assert [(p.l2, p.l3) for p in t.paths] == [(0, 1), (1, 0), (1, 1), (1, 2)]
    R, Nq = 7, 3
    u, x, w = _inputs(t, R, Nq, 2)
    z = oracle.tp_forward(t, x, sh(u, 1), w)
    un = u / np.linalg.norm(u, axis=1, keepdims=True)
    xyz = x[:, [2, 0, 1], :]                     # (y,z,x) -> (x,y,z)
    yzx = [1, 2, 0]
    np.testing.assert_allclose(z[:, 0:3], w[:, 0][:, None] * x, atol=1e-13)
    dot = np.einsum("rkq,rk->rq", xyz, un)
    np.testing.assert_allclose(z[:, 3], w[:, 1] * dot, atol=1e-13)
    cross = np.cross(np.moveaxis(xyz, 1, 2), un[:, None, :])          # [r, q, 3]
    cross = np.moveaxis(cross, 2, 1)[:, yzx, :]
    np.testing.assert_allclose(z[:, 4:7], w[:, 2][:, None] * math.sqrt(1.5) * cross, atol=1e-13)


def test_tp_scalar_case_is_weighted_product():
    t = oracle.table([(0, 1)], 0, 0)
    u, x, w = _inputs(t, 9, 4, 3)
    z = oracle.tp_forward(t, x, sh(u, 0), w)
    np.testing.assert_allclose(z, x * w, atol=1e-15)


@pytest.mark.parametrize("blocks,L2,L3", [(BLOCKS4, 3, 3), ([(0, 1), (1, -1)], 2, 2), (BLOCKS5, 3, 3)])
def test_tp_backward_euler_and_finite_differences(blocks, L2, L3):
    t = oracle.table(blocks, L2, L3)
    R, Nq = 4, 3
    u, x, w = _inputs(t, R, Nq, 4)
    y = sh(u, L2) * 1.3
    dz = np.random.default_rng(9).standard_normal((R, t.D, Nq))
    z = oracle.tp_forward(t, x, y, w)
    dx, dy, dw = oracle.tp_backward(t, x, y, w, dz)
    L = (dz * z).sum()
    # z is linear in each operand: <dz, z> = <dx, x> = <dy, y> = <dw, w>
    for g, a in ((dx, x), (dy, y), (dw, w)):
        np.testing.assert_allclose((g * a).sum(), L, rtol=1e-12)
    # central differences along random directions (exact up to rounding: linear maps)
    rg = np.random.default_rng(10)
    h = 1e-3
    for name, g, a in (("x", dx, x), ("y", dy, y), ("w", dw, w)):
        v = rg.standard_normal(a.shape)
        args = {"x": x, "y": y, "w": w}
        args[name] = a + h * v
        Lp = (dz * oracle.tp_forward(t, args["x"], args["y"], args["w"])).sum()
        args[name] = a - h * v
        Lm = (dz * oracle.tp_forward(t, args["x"], args["y"], args["w"])).sum()
        np.testing.assert_allclose((Lp - Lm) / (2 * h), (g * v).sum(), rtol=1e-9)


def _graph(N, E, seed, empty=2):
    return random_graph(N, E, (90, seed), empty_nodes=empty)


def test_conv_is_scatter_sum_of_edge_products():
    t = oracle.table(BLOCKS4, 3, 3)
    g = _graph(9, 40, 1)
    Nq = 4
    rg = np.random.default_rng(11)
    x = rg.standard_normal((g.n_nodes, t.d1, Nq))
    w = rg.standard_normal((g.n_edges, t.n_paths, Nq))
    y = sh(g.vec, 3)
    scale = 0.37
    m = oracle.conv_forward(t, g.rowptr, g.sender, x, y, w, scale)
    ze = oracle.tp_forward(t, x[g.sender], y, w)
    want = np.zeros((g.n_nodes, t.D, Nq))
    np.add.at(want, g.receiver(), ze)
    np.testing.assert_allclose(m, scale * want, atol=1e-12)
    assert np.all(m[-2:] == 0)          # the two receivers with no edges
    # a subset of receivers gives the same rows
    sub = np.array([5, 0, 3])
    np.testing.assert_allclose(oracle.conv_forward(t, g.rowptr, g.sender, x, y, w, scale, sub),
                               m[sub], atol=0)


def test_conv_scalar_case_is_sparse_matmul():
    """Only (0e, 0 -> 0e): m[:, 0, q] = scale * A_q x[:, 0, q], A_q = CSR(w[:,0,q], sender)."""
    sparse = pytest.importorskip("scipy.sparse")
    t = oracle.table([(0, 1)], 0, 0)
    g = _graph(12, 60, 2, empty=3)
    Nq = 5
    rg = np.random.default_rng(12)
    x = rg.standard_normal((g.n_nodes, 1, Nq))
    w = rg.standard_normal((g.n_edges, 1, Nq))
    m = oracle.conv_forward(t, g.rowptr, g.sender, x, sh(g.vec, 0), w, 0.5)
    for q in range(Nq):
        A = sparse.csr_matrix((w[:, 0, q], g.sender, g.rowptr), shape=(g.n_nodes, g.n_nodes))
        np.testing.assert_allclose(m[:, 0, q], 0.5 * (A @ x[:, 0, q]), atol=1e-13)


def test_conv_equivariance():
    t = oracle.table(BLOCKS4, 3, 3)
    g = _graph(7, 30, 3)
    Nq = 3
    rg = np.random.default_rng(13)
    x = rg.standard_normal((g.n_nodes, t.d1, Nq))
    w = rg.standard_normal((g.n_edges, t.n_paths, Nq))
    R = Rotation.random(random_state=5).as_matrix()
    m = oracle.conv_forward(t, g.rowptr, g.sender, x, sh(g.vec, 3), w, 1.0)
    mr = oracle.conv_forward(t, g.rowptr, g.sender, _rotate_x(t, x, R), sh(g.vec @ R.T, 3), w, 1.0)
    np.testing.assert_allclose(mr, _rotate_z(t, m, R), atol=1e-11)


def test_conv_backward_composition_euler_fd():
    t = oracle.table(BLOCKS4, 3, 3)
    g = _graph(8, 36, 4)
    Nq = 3
    rg = np.random.default_rng(14)
    x = rg.standard_normal((g.n_nodes, t.d1, Nq))
    w = rg.standard_normal((g.n_edges, t.n_paths, Nq))
    y = sh(g.vec, 3)
    dm = rg.standard_normal((g.n_nodes, t.D, Nq))
    scale = 0.8
    dy, dw = oracle.conv_backward_edges(t, g.rowptr, g.sender, x, y, w, dm, scale)
    dx = oracle.conv_backward_dx(t, g.rowptr, g.sender, y, w, dm, scale)
    # composition: per-edge TP backward with dz = scale * dm[receiver], dx scattered to senders
    ex, ey, ew = oracle.tp_backward(t, x[g.sender], y, w, scale * dm[g.receiver()])
    np.testing.assert_allclose(dy, ey, atol=1e-12)
    np.testing.assert_allclose(dw, ew, atol=1e-12)
    want = np.zeros_like(x)
    np.add.at(want, g.sender, ex)
    np.testing.assert_allclose(dx, want, atol=1e-12)
    # Euler identity and finite differences of L = <dm, conv(x, y, w)>
    conv = lambda a, b, c: oracle.conv_forward(t, g.rowptr, g.sender, a, b, c, scale)
    L = (dm * conv(x, y, w)).sum()
    for gr, a in ((dx, x), (dy, y), (dw, w)):
        np.testing.assert_allclose((gr * a).sum(), L, rtol=1e-12)
    v = rg.standard_normal(x.shape)
    fd = ((dm * conv(x + 1e-3 * v, y, w)).sum() - (dm * conv(x - 1e-3 * v, y, w)).sum()) / 2e-3
    np.testing.assert_allclose(fd, (dx * v).sum(), rtol=1e-9)
    # subsets
    sub = np.array([3, 1])
    np.testing.assert_allclose(oracle.conv_backward_dx(t, g.rowptr, g.sender, y, w, dm, scale, sub),
                               dx[sub], atol=0)
    es = np.array([0, 17, 35])
    sy, sw = oracle.conv_backward_edges(t, g.rowptr, g.sender, x, y, w, dm, scale, es)
    np.testing.assert_allclose(sy, dy[es], atol=0)
    np.testing.assert_allclose(sw, dw[es], atol=0)


def test_conv_empty_graph():
    t = oracle.table(BLOCKS4, 3, 3)
    g = _graph(5, 0, 5, empty=0)
    Nq = 2
    x = np.ones((5, t.d1, Nq))
    m = oracle.conv_forward(t, g.rowptr, g.sender, x, np.zeros((0, 16)),
                            np.zeros((0, t.n_paths, Nq)), 1.0)
    assert m.shape == (5, t.D, Nq) and np.all(m == 0)
