"""Radial edge scalars: the per-edge, per-path, per-channel weights w[e, p, q] as a function of
the edge length |r_e| (float64). TEST INFRASTRUCTURE, like the rest of this package.

e3j's notation section (App. E.1, the edge scalars s) says they are "usually" an MLP applied
to a radial embedding of the interatomic distance, projected to the paths and channels of each
edge, and App. A.3 ("Linear mixing") names fusing that scalar mixing into message passing as an
opportunity. The pages fix neither the embedding nor the MLP; the reading taken here is:

  radial embedding  b_n(d) = e_n(d) u(d / r_c),  n = 1..n_basis,
                    e_n(d) = sqrt(2 / r_c) sin(n pi d / r_c) / d   (the Bessel basis: spherical
                    Bessel functions j_0 of the n-th root, orthonormal on [0, r_c] with weight d^2)
                    u(x) = 1 - (p+1)(p+2)/2 x^p + p(p+2) x^(p+1) - p(p+1)/2 x^(p+2) for x < 1,
                    0 beyond (p = 6: the polynomial with u(0) = 1 and u, u', u'' zero at x = 1)
  hidden layer      a_k = sum_n b_n W1[n, k],  h_k = silu(a_k) = a_k / (1 + exp(-a_k))
  output layer      w[p, q] = sum_k h_k W2[k, p, q]

W1 [n_basis, H], W2 [H, P, Nq]; no biases, so an edge at or beyond the cutoff has w = 0. The
cutoff r_c is the graph's. A zero-length vector takes the d -> 0 limit e_n = sqrt(2/r_c) n pi/r_c
and has no gradient (its direction is undefined, as in the harmonics).

The split of this module follows the fused kernels: ``hidden`` gives h[E, H] (the cheap part,
per edge), ``weights`` the full w (what the fused convolution never writes out), and
``hidden_backward`` turns a cotangent dh[E, H] into the gradient with respect to the edge
vectors (forces through the radial weights).
"""
from __future__ import annotations

import numpy as np

P_ENVELOPE = 6


def bessel(d, n_basis: int, r_cut: float):
    """e_n(d), n = 1..n_basis: [len(d), n_basis]."""
    d = np.asarray(d, dtype=np.float64)[:, None]
    k = np.arange(1, n_basis + 1, dtype=np.float64)[None, :] * np.pi / r_cut
    c = np.sqrt(2.0 / r_cut)
    small = d < 1e-12
    safe = np.where(small, 1.0, d)
    return np.where(small, c * k, c * np.sin(k * safe) / safe)


def bessel_grad(d, n_basis: int, r_cut: float):
    """de_n/dd: [len(d), n_basis] (zero at d = 0, where e_n is flat)."""
    d = np.asarray(d, dtype=np.float64)[:, None]
    k = np.arange(1, n_basis + 1, dtype=np.float64)[None, :] * np.pi / r_cut
    c = np.sqrt(2.0 / r_cut)
    small = d < 1e-12
    safe = np.where(small, 1.0, d)
    return np.where(small, 0.0, c * (k * safe * np.cos(k * safe) - np.sin(k * safe)) / (safe * safe))


def envelope(x, p: int = P_ENVELOPE):
    """u(x) for x = d / r_c."""
    x = np.asarray(x, dtype=np.float64)
    u = 1.0 - (p + 1) * (p + 2) / 2.0 * x ** p + p * (p + 2) * x ** (p + 1) - p * (p + 1) / 2.0 * x ** (p + 2)
    return np.where(x < 1.0, u, 0.0)


def envelope_grad(x, p: int = P_ENVELOPE):
    """du/dx."""
    x = np.asarray(x, dtype=np.float64)
    g = (-p * (p + 1) * (p + 2) / 2.0 * x ** (p - 1) + p * (p + 1) * (p + 2) * x ** p
         - p * (p + 1) * (p + 2) / 2.0 * x ** (p + 1))
    return np.where(x < 1.0, g, 0.0)


def basis(d, n_basis: int, r_cut: float):
    """b_n(d) = e_n(d) u(d / r_c): [len(d), n_basis]."""
    d = np.asarray(d, dtype=np.float64)
    return bessel(d, n_basis, r_cut) * envelope(d / r_cut)[:, None]


def basis_grad(d, n_basis: int, r_cut: float):
    """db_n/dd (product rule)."""
    d = np.asarray(d, dtype=np.float64)
    u = envelope(d / r_cut)[:, None]
    du = envelope_grad(d / r_cut)[:, None] / r_cut
    return bessel_grad(d, n_basis, r_cut) * u + bessel(d, n_basis, r_cut) * du


def silu(a):
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def silu_grad(a):
    a = np.asarray(a, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-a))
    return s * (1.0 + a * (1.0 - s))


def lengths(vec):
    vec = np.asarray(vec, dtype=np.float64)
    return np.sqrt(np.sum(vec * vec, axis=1))


def hidden(vec, W1, r_cut: float):
    """h[E, H] = silu(b(|vec|) @ W1)."""
    W1 = np.asarray(W1, dtype=np.float64)
    return silu(basis(lengths(vec), W1.shape[0], r_cut) @ W1)


def weights(vec, W1, W2, r_cut: float):
    """w[E, P, Nq] = sum_k h_k W2[k]."""
    h = hidden(vec, W1, r_cut)
    return np.einsum("ek,kpq->epq", h, np.asarray(W2, dtype=np.float64))


def hidden_from_weights_cotangent(dw, W2):
    """dh[E, H] = sum_{p,q} W2[k, p, q] dw[e, p, q]: the cotangent of the hidden layer."""
    return np.einsum("kpq,epq->ek", np.asarray(W2, dtype=np.float64), np.asarray(dw, dtype=np.float64))


def hidden_backward(vec, W1, r_cut: float, dh):
    """dvec[E, 3]: gradient of sum_{e,k} dh[e,k] h[e,k] with respect to the edge vectors.
    dh/dd = silu'(a) * (b'(d) @ W1); dd/dvec = vec / |vec| (zero for a zero vector)."""
    vec = np.asarray(vec, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    d = lengths(vec)
    nb = W1.shape[0]
    a = basis(d, nb, r_cut) @ W1
    dd = np.sum(np.asarray(dh, dtype=np.float64) * silu_grad(a) * (basis_grad(d, nb, r_cut) @ W1), axis=1)
    unit = np.where(d[:, None] < 1e-12, 0.0, vec / np.where(d < 1e-12, 1.0, d)[:, None])
    return dd[:, None] * unit
