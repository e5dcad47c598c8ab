"""Pins of the generic COO tensor product oracle (oracle/coo.py, e3j App. E.1 Eq. (10)-(11),
Alg. 1).

- a dense einsum over the coefficient tensor assembled from the records (duplicates added);
- with the CG records of a path table it is the CG tensor product of oracle.tp_forward /
  tp_backward (dense per-path CG blocks in plain C loops);
- the backward is the adjoint: <dz, z> = <dx, x> = <dy, y> = <dw, w> (z is linear in each
  operand) and exact directional derivatives of <dz, z> along random directions.
"""
import numpy as np
import pytest

import oracle
from oracle.coo import cg_records, coo_tp_backward, coo_tp_forward


def _random_case(seed, R=7, d1=5, d2=4, D=6, P=3, Nq=3, n=40):
    r = np.random.default_rng(seed)
    recs = np.stack([r.integers(0, D, n), r.integers(0, d1, n), r.integers(0, d2, n), r.integers(0, P, n)], 1)
    recs[1] = recs[0]   # a duplicate record
    c = r.standard_normal(n)
    x, y = r.standard_normal((R, d1, Nq)), r.standard_normal((R, d2))
    w, dz = r.standard_normal((R, P, Nq)), r.standard_normal((R, D, Nq))
    return recs, c, x, y, w, dz, D, r


def test_coo_forward_is_dense_einsum():
    recs, c, x, y, w, dz, D, _ = _random_case(1)
    C = np.zeros((D, x.shape[1], y.shape[1], w.shape[1]))
    np.add.at(C, (recs[:, 0], recs[:, 1], recs[:, 2], recs[:, 3]), c)
    ref = np.einsum("aijp,rpq,riq,rj->raq", C, w, x, y)
    np.testing.assert_allclose(coo_tp_forward(recs, c, x, y, w, D), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("blocks,L2,L3", [([(0, 1), (1, -1), (2, 1)], 3, 3), ([(0, 1), (1, -1)], 2, 2)])
def test_cg_records_give_the_cg_tensor_product(blocks, L2, L3):
    t = oracle.table(blocks, L2, L3)
    recs, c = cg_records(t)
    assert np.all(np.diff(recs[:, 0]) >= 0)
    r = np.random.default_rng(2)
    R, Nq = 9, 4
    x, y = r.standard_normal((R, t.d1, Nq)), r.standard_normal((R, t.d2))
    w, dz = r.standard_normal((R, t.n_paths, Nq)), r.standard_normal((R, t.D, Nq))
    np.testing.assert_allclose(coo_tp_forward(recs, c, x, y, w, t.D), oracle.tp_forward(t, x, y, w), atol=1e-12)
    for got, ref in zip(coo_tp_backward(recs, c, x, y, w, dz), oracle.tp_backward(t, x, y, w, dz)):
        np.testing.assert_allclose(got, ref, atol=1e-12)


def test_coo_backward_is_the_adjoint():
    recs, c, x, y, w, dz, D, r = _random_case(3)
    z = coo_tp_forward(recs, c, x, y, w, D)
    dx, dy, dw = coo_tp_backward(recs, c, x, y, w, dz)
    L = (dz * z).sum()
    for g, a in ((dx, x), (dy, y), (dw, w)):
        np.testing.assert_allclose((g * a).sum(), L, rtol=1e-12)
    # <dz, z> is linear in each operand: a unit step is an exact directional derivative
    for name, g in (("x", dx), ("y", dy), ("w", dw)):
        args = dict(x=x, y=y, w=w)
        v = r.standard_normal(args[name].shape)
        args[name] = args[name] + v
        exact = (dz * coo_tp_forward(recs, c, args["x"], args["y"], args["w"], D)).sum() - L
        np.testing.assert_allclose((g * v).sum(), exact, rtol=1e-10, atol=1e-10)
