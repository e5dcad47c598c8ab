"""Pins of the oracle's radial edge scalars (oracle/radial.py).

e3j, App. E.1 (the edge scalars s: an MLP on a radial embedding of the interatomic distance,
projected to the paths and channels of each edge) and App. A.3 ("Linear mixing": scalar mixing
fused into message passing). The reading (Bessel basis, polynomial envelope, one SiLU hidden
layer) is the oracle's; these tests tie each piece to facts outside it: scipy's spherical
Bessel functions and quadrature, the envelope's defining conditions solved independently,
finite differences, and the forces of the whole radial-weighted convolution.
"""
import numpy as np
import pytest
from scipy import integrate, special
from scipy.spatial.transform import Rotation

import oracle
from oracle import radial
from synth import random_graph

RC = 4.571


def test_bessel_is_scaled_spherical_j0():
    d = np.linspace(0.05, RC, 57)
    nb = 8
    k = np.arange(1, nb + 1) * np.pi / RC
    want = np.sqrt(2 / RC) * k[None, :] * special.spherical_jn(0, k[None, :] * d[:, None])
    assert np.allclose(radial.bessel(d, nb, RC), want, rtol=1e-13, atol=1e-13)
    dwant = np.sqrt(2 / RC) * k[None, :] ** 2 * special.spherical_jn(0, k[None, :] * d[:, None], derivative=True)
    assert np.allclose(radial.bessel_grad(d, nb, RC), dwant, rtol=1e-12, atol=1e-12)
    # the d -> 0 limit
    assert np.allclose(radial.bessel(np.array([0.0]), nb, RC)[0], np.sqrt(2 / RC) * k)


def test_bessel_basis_orthonormal_with_weight_d2():
    nb = 6
    G = np.zeros((nb, nb))
    for n in range(nb):
        for m in range(nb):
            f = lambda d: radial.bessel(np.array([d]), nb, RC)[0, n] * radial.bessel(np.array([d]), nb, RC)[0, m] * d * d
            G[n, m] = integrate.quad(f, 0.0, RC, limit=200)[0]
    assert np.allclose(G, np.eye(nb), atol=1e-9)


def test_envelope_is_the_polynomial_its_conditions_define():
    p = radial.P_ENVELOPE
    # u(x) = 1 + A x^p + B x^(p+1) + C x^(p+2) with u(1) = u'(1) = u''(1) = 0
    M = np.array([[1.0, 1.0, 1.0],
                  [p, p + 1.0, p + 2.0],
                  [p * (p - 1.0), (p + 1.0) * p, (p + 2.0) * (p + 1.0)]])
    A, B, C = np.linalg.solve(M, np.array([-1.0, 0.0, 0.0]))
    x = np.linspace(0, 1, 101)
    assert np.allclose(radial.envelope(x), 1 + A * x ** p + B * x ** (p + 1) + C * x ** (p + 2), atol=1e-13)
    poly = np.polynomial.Polynomial([1.0] + [0.0] * (p - 1) + [A, B, C])
    assert np.allclose(radial.envelope_grad(x[:-1]), poly.deriv()(x[:-1]), atol=1e-12)
    assert radial.envelope(np.array([0.0]))[0] == 1.0
    assert np.all(radial.envelope(np.array([1.0, 1.3])) == 0.0)
    assert np.all(np.diff(radial.envelope(x)) < 0)             # decreasing on (0, 1)
    assert abs(poly.deriv(2)(1.0)) < 1e-9                       # smooth at the cutoff


def test_silu_and_its_gradient():
    a = np.linspace(-12, 12, 97)
    assert np.allclose(radial.silu(a), a * special.expit(a), rtol=1e-14, atol=1e-15)
    h = 1e-6
    fd = (radial.silu(a + h) - radial.silu(a - h)) / (2 * h)
    assert np.allclose(radial.silu_grad(a), fd, rtol=1e-7, atol=1e-9)


def _params(nb=8, H=8, P=5, Nq=6, seed=0):
    r = np.random.default_rng(seed)
    return 2.0 * r.standard_normal((nb, H)), r.standard_normal((H, P, Nq)) / np.sqrt(H * P)


def test_basis_gradient_and_cutoff():
    d = np.linspace(0.3, RC * 0.999, 40)
    h = 1e-6
    fd = (radial.basis(d + h, 8, RC) - radial.basis(d - h, 8, RC)) / (2 * h)
    assert np.allclose(radial.basis_grad(d, 8, RC), fd, rtol=1e-6, atol=1e-9)
    W1, W2 = _params()
    vec = np.array([[RC, 0, 0], [0, RC * 1.2, 0], [0.0, 0.0, 0.0]])
    w = radial.weights(vec[:2], W1, W2, RC)
    assert np.all(w == 0.0)                                      # at and beyond the cutoff
    assert np.all(radial.hidden_backward(vec, W1, RC, np.ones((3, 8)))[2] == 0.0)   # zero vector


def test_weights_are_the_two_layer_network():
    W1, W2 = _params()
    vec = np.random.default_rng(3).standard_normal((30, 3))
    d = np.linalg.norm(vec, axis=1)
    b = radial.basis(d, 8, RC)
    h = (b @ W1) * special.expit(b @ W1)
    want = np.tensordot(h, W2, axes=(1, 0))
    assert np.allclose(radial.weights(vec, W1, W2, RC), want, rtol=1e-13, atol=1e-15)
    # rotation invariance: the weights see only the length
    R = Rotation.random(random_state=4).as_matrix()
    assert np.allclose(radial.weights(vec @ R.T, W1, W2, RC), want, rtol=1e-12, atol=1e-14)


def test_hidden_backward_finite_differences():
    W1, _ = _params()
    rng = np.random.default_rng(5)
    vec = rng.standard_normal((20, 3)) * 1.5
    dh = rng.standard_normal((20, 8))
    g = radial.hidden_backward(vec, W1, RC, dh)
    h = 1e-6
    for c in range(3):
        dv = np.zeros_like(vec)
        dv[:, c] = h
        fd = np.sum(dh * (radial.hidden(vec + dv, W1, RC) - radial.hidden(vec - dv, W1, RC)), axis=1) / (2 * h)
        assert np.allclose(g[:, c], fd, rtol=1e-6, atol=1e-9)


def test_hidden_cotangent_is_the_adjoint_of_the_output_layer():
    _, W2 = _params()
    rng = np.random.default_rng(6)
    h = rng.standard_normal((7, 8))
    dw = rng.standard_normal((7, 5, 6))
    w = np.einsum("ek,kpq->epq", h, W2)
    dh = radial.hidden_from_weights_cotangent(dw, W2)
    assert np.isclose(np.sum(dw * w), np.sum(dh * h), rtol=1e-12)


def test_forces_of_the_radial_weighted_convolution():
    """L(vec) = <dm, conv(x, Y(vec), w(|vec|))>: its gradient through the harmonics (sh_grad of
    the conv's dy) plus through the radial weights (hidden_backward of the conv's dw mapped to
    the hidden layer) equals central finite differences of L in every edge vector."""
    blocks = [(0, 1), (1, -1)]
    t = oracle.table(blocks, 2, 2)
    g = random_graph(9, 40, (97, 1))
    rng = np.random.default_rng(7)
    Nq = 3
    vec = g.vec * 1.3
    x = rng.standard_normal((g.n_nodes, t.d1, Nq))
    dm = rng.standard_normal((g.n_nodes, t.D, Nq))
    W1, W2 = _params(P=t.n_paths, Nq=Nq, seed=8)
    scale = 0.7

    def L(v):
        y = oracle.sh(v, 2)
        w = radial.weights(v, W1, W2, RC)
        return float(np.sum(dm * oracle.conv_forward(t, g.rowptr, g.sender, x, y, w, scale)))

    y = oracle.sh(vec, 2)
    w = radial.weights(vec, W1, W2, RC)
    dy, dw = oracle.conv_backward_edges(t, g.rowptr, g.sender, x, y, w, dm, scale)
    grad = oracle.sh_grad(vec, 2, dy) + radial.hidden_backward(vec, W1, RC, radial.hidden_from_weights_cotangent(dw, W2))
    h = 1e-6
    for e in (0, 7, 19, 39):
        for c in range(3):
            vp, vm = vec.copy(), vec.copy()
            vp[e, c] += h
            vm[e, c] -= h
            fd = (L(vp) - L(vm)) / (2 * h)
            assert np.isclose(grad[e, c], fd, rtol=1e-6, atol=1e-8), (e, c, grad[e, c], fd)
