"""Oracle: the generic sparse-coefficient tensor product (arbitrary bilinear map with per-path
channel weights), float64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows "e3j: An efficient and open-source backend for Euclidean equivariant operations on
GPU and TPU", App. E.1 Eq. (10)-(11) and Alg. 1: the coefficient tensor C is a list of COO
records (i0, i1, i2, path, c) and, per row r and channel q,

    z[r, i0, q] = sum over records with that i0 of  c * w[r, path, q] * x[r, i1, q] * y[r, i2]

(y has no channel axis, the same reading as the CG tensor product). Duplicate records add.
Any coefficient list is allowed: the Clebsch-Gordan product is the case where the records
are the nonzero CG entries of each path. The backward is the exact adjoint:
    dx[r, i1, q] += c w[r,p,q] y[r,i2] dz[r,i0,q];  dw[r, p, q] += c x[r,i1,q] y[r,i2] dz[r,i0,q]
    dy[r, i2]    += sum_q c w[r,p,q] x[r,i1,q] dz[r,i0,q].
"""
from __future__ import annotations

import numpy as np


def coo_tp_forward(recs, c, x, y, w, D: int):
    """recs: int [n, 4] rows (i0, i1, i2, path); c: [n]; x [R, d1, Nq], y [R, d2],
    w [R, P, Nq] -> z [R, D, Nq]."""
    x, y, w = (np.asarray(a, dtype=np.float64) for a in (x, y, w))
    z = np.zeros((x.shape[0], D, x.shape[2]))
    for (i0, i1, i2, p), ck in zip(np.asarray(recs), np.asarray(c, dtype=np.float64)):
        z[:, i0, :] += ck * w[:, p, :] * x[:, i1, :] * y[:, i2, None]
    return z


def coo_tp_backward(recs, c, x, y, w, dz):
    """(dx, dy, dw) for the same records."""
    x, y, w, dz = (np.asarray(a, dtype=np.float64) for a in (x, y, w, dz))
    dx, dy, dw = np.zeros_like(x), np.zeros_like(y), np.zeros_like(w)
    for (i0, i1, i2, p), ck in zip(np.asarray(recs), np.asarray(c, dtype=np.float64)):
        dx[:, i1, :] += ck * w[:, p, :] * y[:, i2, None] * dz[:, i0, :]
        dw[:, p, :] += ck * x[:, i1, :] * y[:, i2, None] * dz[:, i0, :]
        dy[:, i2] += ck * (w[:, p, :] * x[:, i1, :] * dz[:, i0, :]).sum(1)
    return dx, dy, dw


def cg_records(table):
    """The CG tensor product of a path table as COO records (the nonzero entries of each
    path's CG block, output index = the block's row), sorted by i0."""
    from .cg import cg_block
    recs, cs = [], []
    for k, p in enumerate(table.paths):
        C = cg_block(p.l1, p.l2, p.l3)
        for m1, m2, m3 in zip(*np.nonzero(np.abs(C) > 1e-12)):
            recs.append((p.zoff + m3, p.xoff + m1, p.yoff + m2, k))
            cs.append(C[m1, m2, m3])
    recs, cs = np.array(recs, dtype=np.int32).reshape(-1, 4), np.array(cs)
    order = np.argsort(recs[:, 0], kind="stable")
    return recs[order], cs[order]
