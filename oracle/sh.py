"""Oracle: real spherical harmonics Y_l(u), l <= 3, component normalisation.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this package; only
tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg use it.

Follows "e3j: An efficient and open-source backend for Euclidean equivariant operations on
GPU and TPU", App. A.3 Eq. (4) (Y_l = (Y_lm)_{m=-l..l}, concatenated over l = 0..lmax) and
App. G.1 (harmonic polynomials, the degree-l homogeneous harmonic polynomials of x, y, z).

Reading of the pages (they name "real harmonics" but print only the complex top-spin form
Y_l^{+-l} = c_l (x + i y)^l): the textbook real basis, m = -l..l, m < 0 the sin-type and
m > 0 the cos-type combinations, no Condon-Shortley sign, scaled by sqrt(4 pi) so that
sum_m Y_lm(u)^2 = 2l + 1 on the unit sphere ("component" normalisation). For l = 1 this is
sqrt(3) (y, z, x). The polynomials are written in homogeneous form, so Y_l(0) = 0 for
l > 0, and are evaluated at u = r / |r| (u = 0 when |r| < 1e-12).

Each Y_lm is stored as {(a, b, c): coefficient} for the monomial x^a y^b z^c; the CG oracle
differentiates the same polynomials to get the rotation generators.
"""
from __future__ import annotations

import math

import numpy as np

LMAX = 3

_s3, _s5, _s7 = math.sqrt(3), math.sqrt(5), math.sqrt(7)
_s15, _s42, _s70, _s105 = math.sqrt(15), math.sqrt(42), math.sqrt(70), math.sqrt(105)

# POLY[l][m + l] = {(a, b, c): coef} for x^a y^b z^c
POLY: list[list[dict[tuple[int, int, int], float]]] = [
    [{(0, 0, 0): 1.0}],
    [{(0, 1, 0): _s3}, {(0, 0, 1): _s3}, {(1, 0, 0): _s3}],
    [
        {(1, 1, 0): _s15},                                            # xy
        {(0, 1, 1): _s15},                                            # yz
        {(0, 0, 2): _s5, (2, 0, 0): -_s5 / 2, (0, 2, 0): -_s5 / 2},  # (2z^2 - x^2 - y^2)/2
        {(1, 0, 1): _s15},                                            # xz
        {(2, 0, 0): _s15 / 2, (0, 2, 0): -_s15 / 2},                  # (x^2 - y^2)/2
    ],
    [
        {(2, 1, 0): 3 * _s70 / 4, (0, 3, 0): -_s70 / 4},              # y(3x^2 - y^2)
        {(1, 1, 1): _s105},                                           # xyz
        {(0, 1, 2): _s42, (2, 1, 0): -_s42 / 4, (0, 3, 0): -_s42 / 4},  # y(4z^2 - x^2 - y^2)
        {(0, 0, 3): _s7, (2, 0, 1): -3 * _s7 / 2, (0, 2, 1): -3 * _s7 / 2},  # z(2z^2-3x^2-3y^2)/2
        {(1, 0, 2): _s42, (3, 0, 0): -_s42 / 4, (1, 2, 0): -_s42 / 4},  # x(4z^2 - x^2 - y^2)
        {(2, 0, 1): _s105 / 2, (0, 2, 1): -_s105 / 2},                # z(x^2 - y^2)
        {(3, 0, 0): _s70 / 4, (1, 2, 0): -3 * _s70 / 4},              # x(x^2 - 3y^2)
    ],
]


def sh_l(u: np.ndarray, l: int) -> np.ndarray:
    """Y_l at the rows of u [n,3] (used as given, not normalised): [n, 2l+1] float64."""
    u = np.asarray(u, dtype=np.float64)
    x, y, z = u[:, 0], u[:, 1], u[:, 2]
    out = np.zeros((u.shape[0], 2 * l + 1))
    for i, poly in enumerate(POLY[l]):
        for (a, b, c), k in poly.items():
            out[:, i] += k * x ** a * y ** b * z ** c
    return out


def normalise(vec: np.ndarray) -> np.ndarray:
    vec = np.asarray(vec, dtype=np.float64)
    n = np.linalg.norm(vec, axis=1, keepdims=True)
    u = np.zeros_like(vec)
    ok = n[:, 0] >= 1e-12
    u[ok] = vec[ok] / n[ok]
    return u


def sh(vec: np.ndarray, lmax: int) -> np.ndarray:
    """y[n, (lmax+1)^2] = concat_l Y_l(vec / |vec|), float64 (App. A.3 Eq. 4)."""
    if not 0 <= lmax <= LMAX:
        raise ValueError("lmax must be in 0..3")
    u = normalise(vec)
    return np.concatenate([sh_l(u, l) for l in range(lmax + 1)], axis=1)


def _poly_grad(poly: dict, u: np.ndarray) -> np.ndarray:
    """Gradient of a polynomial {(a,b,c): k} at the rows of u: [n, 3]."""
    x, y, z = u[:, 0], u[:, 1], u[:, 2]
    g = np.zeros((u.shape[0], 3))
    for (a, b, c), k in poly.items():
        if a:
            g[:, 0] += k * a * x ** (a - 1) * y ** b * z ** c
        if b:
            g[:, 1] += k * b * x ** a * y ** (b - 1) * z ** c
        if c:
            g[:, 2] += k * c * x ** a * y ** b * z ** (c - 1)
    return g


def sh_grad(vec: np.ndarray, lmax: int, dy: np.ndarray) -> np.ndarray:
    """dvec[n,3] = sum_{l,m} dy[n, l^2 + l + m] dY_lm(vec/|vec|)/dvec (the VJP of sh()).

    Y_lm(u) is the degree-l homogeneous polynomial P_lm at u = r/|r|, so by the chain rule
    and Euler's identity grad P . u = l P:  dY/dr = (grad P(u) - l P(u) u) / |r|.
    Zero where |r| < 1e-12 (Y is taken constant there)."""
    vec = np.asarray(vec, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = np.linalg.norm(vec, axis=1)
    ok = r >= 1e-12
    u = normalise(vec)
    g = np.zeros_like(vec)
    euler = np.zeros(vec.shape[0])
    for l in range(lmax + 1):
        for i, poly in enumerate(POLY[l]):
            d = dy[:, l * l + i]
            g += d[:, None] * _poly_grad(poly, u)
            euler += d * l * sh_l(u, l)[:, i]
    out = np.zeros_like(vec)
    out[ok] = (g[ok] - euler[ok, None] * u[ok]) / r[ok, None]
    return out
