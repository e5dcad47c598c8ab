"""Oracle: real Clebsch-Gordan blocks C[m1, m2, m3] for (l1, l2) -> l3, l <= 3 (float64).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Definition used ("e3j ...", App. A.3 Eq. (6) and App. G.2): the CG block of a path is the
(unique up to scale) bilinear map z = C(a, b), z_m3 = sum C[m1,m2,m3] a_m1 b_m2, that is
equivariant, C(D^l1(R) a, D^l2(R) b) = D^l3(R) C(a, b) for every rotation R, where D^l(R) is
the matrix with Y_l(R u) = D^l(R) Y_l(u) for the real harmonics of oracle/sh.py.

Construction (independent of any CG formula): differentiate that condition at R = 1. For
the three axes k the infinitesimal rotation acts on functions as L_x = y d/dz - z d/dy,
L_y = z d/dx - x d/dz, L_z = x d/dy - y d/dx; applying L_k to the polynomials of oracle/sh.py
and expanding in the same basis gives Gamma_k^l with L_k Y_lm = sum_m' Gamma_k^l[m, m'] Y_lm'.
C then spans the null space of

    sum_a Gamma1[a, m1] C[a, m2, m3] + sum_b Gamma2[b, m2] C[m1, b, m3]
        - sum_c Gamma3[m3, c] C[m1, m2, c] = 0     for k = x, y, z,

found with an SVD. Normalisation (App. G.2 builds unit eigenvectors |L M>): for every m3,
sum_{m1,m2} C[m1,m2,m3]^2 = 1. Sign (the pages fix none): the first entry of C in row-major
(m1, m2, m3) order whose magnitude exceeds 1e-9 max|C| is positive.
"""
from __future__ import annotations

from functools import lru_cache

import numpy as np

from .sh import POLY


def _poly_apply_L(poly: dict, k: int) -> dict:
    """L_k applied to a polynomial {(a,b,c): coef}."""
    out: dict = {}

    def add(mono, c):
        if c != 0.0:
            out[mono] = out.get(mono, 0.0) + c

    for (a, b, c), coef in poly.items():
        # derivative helpers: d/dx x^a = a x^(a-1)
        if k == 0:   # y d/dz - z d/dy
            if c > 0:
                add((a, b + 1, c - 1), coef * c)
            if b > 0:
                add((a, b - 1, c + 1), -coef * b)
        elif k == 1:  # z d/dx - x d/dz
            if a > 0:
                add((a - 1, b, c + 1), coef * a)
            if c > 0:
                add((a + 1, b, c - 1), -coef * c)
        else:        # x d/dy - y d/dx
            if b > 0:
                add((a + 1, b - 1, c), coef * b)
            if a > 0:
                add((a - 1, b + 1, c), -coef * a)
    return out


def _monomials(l: int):
    return [(a, b, l - a - b) for a in range(l + 1) for b in range(l + 1 - a)]


@lru_cache(maxsize=None)
def generators(l: int) -> np.ndarray:
    """Gamma[k] (3, 2l+1, 2l+1): L_k Y_lm = sum_m' Gamma[k][m, m'] Y_lm'."""
    monos = _monomials(l)
    idx = {m: i for i, m in enumerate(monos)}
    n = 2 * l + 1
    B = np.zeros((len(monos), n))          # basis polynomials as columns
    for j, poly in enumerate(POLY[l]):
        for mono, c in poly.items():
            B[idx[mono], j] = c
    G = np.zeros((3, n, n))
    for k in range(3):
        for m in range(n):
            img = _poly_apply_L(POLY[l][m], k)
            v = np.zeros(len(monos))
            for mono, c in img.items():
                v[idx[mono]] = c
            coef, res, *_ = np.linalg.lstsq(B, v, rcond=None)
            if np.abs(B @ coef - v).max() > 1e-10:
                raise RuntimeError("harmonic space not invariant under L")
            G[k, m, :] = coef
    return G


@lru_cache(maxsize=None)
def cg_block(l1: int, l2: int, l3: int) -> np.ndarray:
    """C[2l1+1, 2l2+1, 2l3+1] float64; all zeros when the triangle rule fails."""
    n1, n2, n3 = 2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        return np.zeros((n1, n2, n3))
    G1, G2, G3 = generators(l1), generators(l2), generators(l3)
    I1, I2, I3 = np.eye(n1), np.eye(n2), np.eye(n3)
    rows = []
    for k in range(3):
        M = (np.kron(np.kron(G1[k].T, I2), I3) + np.kron(np.kron(I1, G2[k].T), I3)
             - np.kron(np.kron(I1, I2), G3[k]))
        rows.append(M)
    A = np.concatenate(rows, axis=0)
    _, s, vt = np.linalg.svd(A)
    # vt has n1 n2 n3 rows; singular values beyond len(s) are zero too
    tol = 1e-9 * max(1.0, s.max())
    svals = np.concatenate([s, np.zeros(vt.shape[0] - s.size)])
    null = vt[svals < tol]
    if null.shape[0] != 1:
        raise RuntimeError(f"null space of ({l1},{l2},{l3}) has dim {null.shape[0]}")
    C = null[0].reshape(n1, n2, n3)
    C = C * np.sqrt(n3 / np.sum(C * C))
    flat = C.reshape(-1)
    big = np.abs(flat) > 1e-9 * np.abs(flat).max()
    first = np.nonzero(big)[0][0]
    if flat[first] < 0:
        C = -C
    C[np.abs(C) < 1e-10] = 0.0   # SVD noise is ~1e-14; true entries are >= 0.1
    return C
