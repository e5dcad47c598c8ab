"""Pins of the oracle's real spherical harmonics (oracle/sh.py) to facts outside it.

"e3j ...", App. A.2-A.3 Eq. (4) and App. G.1: Y_l is the bank of 2l+1 degree-l harmonic
polynomials, rotation-equivariant, with parity (-1)^l.
"""
import math

import numpy as np
import pytest

from oracle.sh import POLY, sh, sh_l


def _units(n, seed):
    g = np.random.default_rng(seed).standard_normal((n, 3))
    return g / np.linalg.norm(g, axis=1, keepdims=True)


def _real_sh_scipy(l, u):
    """Textbook real SH from scipy's complex Y_l^m (Condon-Shortley phase included):
    m > 0: sqrt2 (-1)^m Re Y_l^m, m < 0: sqrt2 (-1)^m Im Y_l^|m|, m = 0: Y_l^0; times
    sqrt(4 pi) for component normalisation."""
    sp = pytest.importorskip("scipy.special")
    theta = np.arccos(np.clip(u[:, 2], -1, 1))          # polar
    phi = np.arctan2(u[:, 1], u[:, 0])                  # azimuth
    if hasattr(sp, "sph_harm_y"):
        Y = lambda m: sp.sph_harm_y(l, m, theta, phi)
    else:  # older scipy: sph_harm(m, l, azimuth, polar)
        Y = lambda m: sp.sph_harm(m, l, phi, theta)
    out = np.zeros((u.shape[0], 2 * l + 1))
    for m in range(-l, l + 1):
        if m > 0:
            v = math.sqrt(2) * (-1) ** m * Y(m).real
        elif m < 0:
            v = math.sqrt(2) * (-1) ** m * Y(-m).imag
        else:
            v = Y(0).real
        out[:, m + l] = v * math.sqrt(4 * math.pi)
    return out


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_matches_library_associated_legendre(l):
    u = _units(64, 1)
    np.testing.assert_allclose(sh_l(u, l), _real_sh_scipy(l, u), atol=1e-12)


def test_l1_is_sqrt3_yzx():
    u = _units(16, 2)
    np.testing.assert_allclose(sh_l(u, 1), math.sqrt(3) * u[:, [1, 2, 0]], atol=1e-15)


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_component_normalisation(l):
    u = _units(100, 3)
    np.testing.assert_allclose((sh_l(u, l) ** 2).sum(1), 2 * l + 1, rtol=1e-13)


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_addition_theorem(l):
    """sum_m Y_lm(u) Y_lm(v) = (2l+1) P_l(u.v), P_l from numpy's Legendre series."""
    u, v = _units(50, 4), _units(50, 5)
    lhs = (sh_l(u, l) * sh_l(v, l)).sum(1)
    coef = np.zeros(l + 1); coef[l] = 1
    rhs = (2 * l + 1) * np.polynomial.legendre.legval((u * v).sum(1), coef)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_parity(l):
    u = _units(20, 6)
    np.testing.assert_allclose(sh_l(-u, l), (-1) ** l * sh_l(u, l), atol=1e-14)


@pytest.mark.parametrize("l", [1, 2, 3])
def test_harmonic_and_homogeneous(l):
    """Laplacian of every polynomial is zero (exact, on the monomial coefficients)."""
    for poly in POLY[l]:
        lap = {}
        for (a, b, c), k in poly.items():
            assert a + b + c == l
            for i, e in enumerate((a, b, c)):
                if e >= 2:
                    mono = [a, b, c]; mono[i] -= 2
                    lap[tuple(mono)] = lap.get(tuple(mono), 0.0) + k * e * (e - 1)
        assert all(abs(v) < 1e-12 for v in lap.values())


def test_axis_values_and_zero_vector():
    z = np.array([[0.0, 0.0, 2.5]])
    y = sh(z, 3)[0]
    for l in range(4):
        blk = y[l * l:(l + 1) ** 2]
        want = np.zeros(2 * l + 1); want[l] = math.sqrt(2 * l + 1)   # only m = 0 survives
        np.testing.assert_allclose(blk, want, atol=1e-14)
    y0 = sh(np.zeros((1, 3)), 3)[0]
    assert y0[0] == 1.0 and np.all(y0[1:] == 0.0)


def test_rotation_equivariance_via_lstsq():
    """Y_l(R u) = D^l(R) Y_l(u) has an orthogonal solution D (a representation)."""
    from scipy.spatial.transform import Rotation
    R = Rotation.random(random_state=7).as_matrix()
    u = _units(200, 8)
    for l in range(4):
        A, B = sh_l(u, l), sh_l(u @ R.T, l)
        D = np.linalg.lstsq(A, B, rcond=None)[0].T
        np.testing.assert_allclose(A @ D.T, B, atol=1e-12)
        np.testing.assert_allclose(D @ D.T, np.eye(2 * l + 1), atol=1e-12)


@pytest.mark.parametrize("lmax", [0, 1, 2, 3])
def test_sh_grad_finite_differences(lmax):
    """sh_grad is the VJP of sh: <dvec, v> = d/dt <dy, sh(r + t v)> (central differences)."""
    from oracle.sh import sh_grad
    rng = np.random.default_rng(30 + lmax)
    r = rng.standard_normal((25, 3)) * rng.uniform(0.3, 3.0, (25, 1))
    dy = rng.standard_normal((25, (lmax + 1) ** 2))
    v = rng.standard_normal((25, 3))
    h = 1e-6
    fd = ((dy * sh(r + h * v, lmax)).sum(1) - (dy * sh(r - h * v, lmax)).sum(1)) / (2 * h)
    np.testing.assert_allclose((sh_grad(r, lmax, dy) * v).sum(1), fd, rtol=1e-6, atol=1e-8)


def test_sh_grad_radial_scaling_rotation():
    from scipy.spatial.transform import Rotation
    from oracle.sh import sh_grad
    rng = np.random.default_rng(40)
    r = rng.standard_normal((30, 3))
    dy = rng.standard_normal((30, 16))
    g = sh_grad(r, 3, dy)
    # Y depends on the direction only: no radial component, 1/s under r -> s r
    np.testing.assert_allclose((g * r).sum(1), 0.0, atol=1e-12)
    np.testing.assert_allclose(sh_grad(2.5 * r, 3, dy), g / 2.5, atol=1e-12)
    # rotating r and the cotangent (by the SH representation) rotates the gradient
    R = Rotation.random(random_state=4).as_matrix()
    u = rng.standard_normal((200, 3))
    dyr = np.zeros_like(dy)
    for l in range(4):
        D = np.linalg.lstsq(sh_l(u, l), sh_l(u @ R.T, l), rcond=None)[0].T
        dyr[:, l * l:(l + 1) ** 2] = dy[:, l * l:(l + 1) ** 2] @ D.T
    np.testing.assert_allclose(sh_grad(r @ R.T, 3, dyr), g @ R.T, atol=1e-11)
    # zero vector: zero gradient
    assert np.all(sh_grad(np.zeros((1, 3)), 3, np.ones((1, 16))) == 0.0)
