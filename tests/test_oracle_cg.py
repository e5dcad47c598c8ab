"""Pins of the oracle's CG blocks (oracle/cg.py) and path tables (oracle/paths.py).

"e3j ...", App. A.3 Eq. (6) (CG tensor product paths L = |l-l'|..l+l'), App. B.1 (parity
rule) and App. G.2 (CG as unit eigenvectors |L M>).
"""
import math

import numpy as np
import pytest
from scipy.spatial.transform import Rotation

from oracle.cg import cg_block
from oracle.paths import make_table
from oracle.sh import sh_l

TRI = [(l1, l2, l3) for l1 in range(4) for l2 in range(4)
       for l3 in range(abs(l1 - l2), min(3, l1 + l2) + 1)]


def _units(n, seed):
    g = np.random.default_rng(seed).standard_normal((n, 3))
    return g / np.linalg.norm(g, axis=1, keepdims=True)


def _wigner_from_sh(R, l):
    u = _units(200, 11)
    return np.linalg.lstsq(sh_l(u, l), sh_l(u @ R.T, l), rcond=None)[0].T


@pytest.mark.parametrize("l1,l2", [(a, b) for a in range(4) for b in range(4)])
def test_orthogonality(l1, l2):
    """Columns (l3, m3) of the stacked blocks are orthonormal; when every l3 <= 3 the
    stacked matrix is square, i.e. an orthogonal change of basis of l1 (x) l2."""
    cols = [cg_block(l1, l2, l3).reshape(-1, 2 * l3 + 1)
            for l3 in range(abs(l1 - l2), min(3, l1 + l2) + 1)]
    M = np.concatenate(cols, axis=1)
    np.testing.assert_allclose(M.T @ M, np.eye(M.shape[1]), atol=1e-12)
    if l1 + l2 <= 3:
        assert M.shape[0] == M.shape[1]
        np.testing.assert_allclose(M @ M.T, np.eye(M.shape[0]), atol=1e-12)


@pytest.mark.parametrize("l1,l2,l3", TRI)
def test_equivariance_finite_rotation(l1, l2, l3):
    R = Rotation.random(random_state=l1 * 16 + l2 * 4 + l3).as_matrix()
    D1, D2, D3 = (_wigner_from_sh(R, l) for l in (l1, l2, l3))
    C = cg_block(l1, l2, l3)
    g = np.random.default_rng(5)
    a, b = g.standard_normal(2 * l1 + 1), g.standard_normal(2 * l2 + 1)
    lhs = np.einsum("ijk,i,j->k", C, D1 @ a, D2 @ b)
    rhs = D3 @ np.einsum("ijk,i,j->k", C, a, b)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)


@pytest.mark.parametrize("l1,l2,l3", TRI)
def test_sign_rule(l1, l2, l3):
    flat = cg_block(l1, l2, l3).reshape(-1)
    assert flat[np.nonzero(flat)[0][0]] > 0


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_scalar_times_irrep_is_identity(l):
    np.testing.assert_allclose(cg_block(0, l, l)[0], np.eye(2 * l + 1), atol=1e-14)
    np.testing.assert_allclose(cg_block(l, 0, l)[:, 0, :], np.eye(2 * l + 1), atol=1e-14)


def test_dot_and_cross():
    g = np.random.default_rng(3)
    a, b = g.standard_normal(3), g.standard_normal(3)          # (x, y, z)
    yzx = [1, 2, 0]
    A, B = a[yzx], b[yzx]
    dot = np.einsum("ijk,i,j->k", cg_block(1, 1, 0), A, B)
    np.testing.assert_allclose(dot, [np.dot(a, b) / math.sqrt(3)], atol=1e-14)
    cross = np.einsum("ijk,i,j->k", cg_block(1, 1, 1), A, B)
    np.testing.assert_allclose(cross, np.cross(a, b)[yzx] / math.sqrt(2), atol=1e-14)


@pytest.mark.parametrize("l1,l2,l3", [t for t in TRI if sum(t) % 2 == 0])
def test_product_of_harmonics(l1, l2, l3):
    """For l1+l2+l3 even, C(Y_l1(u), Y_l2(u)) = k Y_l3(u) with
    |k| = sqrt((2l1+1)(2l2+1)/(2l3+1)) |<l1 0 l2 0 | l3 0>| (sympy's CG)."""
    wig = pytest.importorskip("sympy.physics.wigner")
    u = _units(40, 9)
    lhs = np.einsum("ijk,ni,nj->nk", cg_block(l1, l2, l3), sh_l(u, l1), sh_l(u, l2))
    Y3 = sh_l(u, l3)
    k = (lhs * Y3).sum() / (Y3 * Y3).sum()
    np.testing.assert_allclose(lhs, k * Y3, atol=1e-12)
    cg00 = float(wig.clebsch_gordan(l1, l2, l3, 0, 0, 0))
    assert abs(abs(k) - math.sqrt((2 * l1 + 1) * (2 * l2 + 1) / (2 * l3 + 1)) * abs(cg00)) < 1e-12


def test_paths_small_workload():
    """x = 0e+1o, SH l <= 2, outputs l <= 2: the triangles and their parities."""
    t = make_table([(0, 1), (1, -1)], 2, 2)
    got = [(p.xblock, p.l2, p.l3, p.p3) for p in t.paths]
    want = [(0, 0, 0, 1), (0, 1, 1, -1), (0, 2, 2, 1),
            (1, 0, 1, -1), (1, 1, 0, 1), (1, 1, 1, 1), (1, 1, 2, 1), (1, 2, 1, -1), (1, 2, 2, -1)]
    assert got == want
    assert t.out_blocks == [(0, 1), (1, -1), (1, 1), (2, 1), (2, -1)]
    assert (t.d1, t.d2, t.D) == (4, 9, 17)
    pp = make_table([(0, 1), (1, -1)], 2, 2, per_path=True)
    assert pp.D == sum(2 * p.l3 + 1 for p in pp.paths)


@pytest.mark.parametrize("blocks,L2,L3,P,D", [
    ([(0, 1), (1, -1), (2, 1)], 3, 3, 24, 31),
    ([(0, 1), (1, -1)], 3, 3, 13, 31),
    ([(0, 1), (1, -1), (2, 1), (3, -1)], 3, 3, 34, 31),
])
def test_path_counts(blocks, L2, L3, P, D):
    t = make_table(blocks, L2, L3)
    assert (t.n_paths, t.D) == (P, D)
    # every output parity equals p1 (-1)^l2
    for p in t.paths:
        assert p.p3 == p.p1 * (-1) ** p.l2
        assert t.out_blocks[p.out_block] == (p.l3, p.p3)
