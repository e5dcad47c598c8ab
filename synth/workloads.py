"""The five seeded workloads (shapes, sizes and value distributions) and small variants.

Each workload names the irreps of the node/row features x, the SH degree of y, the largest
output degree, the channel count and the problem size. ``make_tp`` / ``make_conv`` return
plain numpy inputs; nothing here computes spherical harmonics or tensor products.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import (STREAM_GRAD, STREAM_POS, STREAM_RADIAL, STREAM_W, STREAM_X, Graph, box_graph, normal_rows,
               rng, unit_vectors)


def parse_irreps(s: str) -> tuple[int, list[tuple[int, int]]]:
    """'128x0e+128x1o' -> (128, [(0, +1), (1, -1)]). Uniform multiplicity only."""
    mul = None
    blocks = []
    for term in s.split("+"):
        m, ir = term.strip().split("x")
        m = int(m)
        if mul is None:
            mul = m
        elif m != mul:
            raise ValueError("uniform multiplicity required")
        l = int(ir[:-1])
        p = {"e": 1, "o": -1}[ir[-1]]
        blocks.append((l, p))
    return mul, blocks


@dataclass(frozen=True)
class Workload:
    wid: int                 # seed namespace
    name: str
    kind: str                # 'tp' or 'conv'
    irreps_x: str
    sh_lmax: int
    out_lmax: int
    rows: int = 0            # tp rows
    n_atoms: int = 0         # conv nodes
    degree: float = 0.0      # conv target average degree (cutoff from density)
    cutoff: float | None = None
    w_unit_std: bool = False  # True: w ~ N(0,1); False: N(0,1)/sqrt(P)

    @property
    def mul(self) -> int:
        return parse_irreps(self.irreps_x)[0]

    @property
    def blocks(self):
        return parse_irreps(self.irreps_x)[1]

    @property
    def d1(self) -> int:
        return sum(2 * l + 1 for l, _ in self.blocks)

    @property
    def d2(self) -> int:
        return (self.sh_lmax + 1) ** 2


WORKLOADS = {
    1: Workload(1, "tp-small: 1024 rows, 16x0e+16x1o, SH l<=2, out l<=2", "tp",
                "16x0e+16x1o", 2, 2, rows=1024, w_unit_std=True),
    2: Workload(2, "tp-batched: 200000 rows, 128x0e+128x1o+128x2e, SH l<=3, out l<=3", "tp",
                "128x0e+128x1o+128x2e", 3, 3, rows=200_000),
    3: Workload(3, "conv: 4096 atoms, rc 5 A, 128x0e+128x1o, SH l<=3, out l<=3", "conv",
                "128x0e+128x1o", 3, 3, n_atoms=4096, cutoff=5.0),
    4: Workload(4, "conv-mace: 64000 atoms, ~40 nbrs, 128x0e+128x1o+128x2e, SH l<=3, out l<=3", "conv",
                "128x0e+128x1o+128x2e", 3, 3, n_atoms=64_000, degree=40.0),
    5: Workload(5, "conv-highl: 100000 atoms, ~30 nbrs, 8x0e+8x1o+8x2e+8x3o, SH l<=3, out l<=3", "conv",
                "8x0e+8x1o+8x2e+8x3o", 3, 3, n_atoms=100_000, degree=30.0),
}


def weight_scale(w: Workload, n_paths: int) -> float:
    """Standard deviation of the weights: 1, or 1/sqrt(P) for P paths (the caller supplies P,
    which the method's path table defines)."""
    return 1.0 if w.w_unit_std else 1.0 / math.sqrt(n_paths)


def make_tp(w: Workload, n_paths: int, rows: int | None = None, row_ids: np.ndarray | None = None):
    """TP inputs: unit vectors u[R,3] (y = SH(u)), x[R,d1,mul], w[R,P,mul], dz draws are
    separate (``make_grad``). row_ids selects rows of the full-size workload."""
    R = w.rows if rows is None else rows
    P = n_paths
    if row_ids is None:
        u = unit_vectors(R, (w.wid, STREAM_POS))
        x = normal_rows(R, (w.d1, w.mul), (w.wid, STREAM_X))
        ww = normal_rows(R, (P, w.mul), (w.wid, STREAM_W), weight_scale(w, P))
    else:
        u = unit_vectors(R, (w.wid, STREAM_POS))[row_ids]
        x = normal_rows(R, (w.d1, w.mul), (w.wid, STREAM_X), rows=row_ids)
        ww = normal_rows(R, (P, w.mul), (w.wid, STREAM_W), weight_scale(w, P), rows=row_ids)
    return u, x, ww


def make_grad(w: Workload, n: int, D: int, row_ids: np.ndarray | None = None) -> np.ndarray:
    return normal_rows(n, (D, w.mul), (w.wid, STREAM_GRAD), rows=row_ids)


def make_graph(w: Workload, n_atoms: int | None = None, order: str = "cell") -> Graph:
    N = w.n_atoms if n_atoms is None else n_atoms
    if w.cutoff is not None:
        return box_graph(w.wid, N, cutoff=w.cutoff, order=order)
    return box_graph(w.wid, N, degree=w.degree, order=order)


def make_conv(w: Workload, g: Graph, n_paths: int, edge_ids: np.ndarray | None = None):
    """Conv inputs for graph g: x[N,d1,mul], w[E,P,mul] (or only the rows edge_ids)."""
    P = n_paths
    x = normal_rows(g.n_nodes, (w.d1, w.mul), (w.wid, STREAM_X))
    ww = normal_rows(g.n_edges, (P, w.mul), (w.wid, STREAM_W), weight_scale(w, P), rows=edge_ids)
    return x, ww


def make_radial(w: Workload, n_paths: int, n_basis: int = 8, hidden: int = 8):
    """Parameters of the radial network (float32): W1[n_basis, hidden] ~ N(0, 2^2) and
    W2[hidden, P, mul] ~ N(0, 1/(hidden P)), so that the weights it produces have roughly the
    spread of the drawn ones."""
    r = rng(w.wid, STREAM_RADIAL)
    W1 = (2.0 * r.standard_normal((n_basis, hidden))).astype(np.float32)
    W2 = (r.standard_normal((hidden, n_paths, w.mul)) / math.sqrt(hidden * n_paths)).astype(np.float32)
    return W1, W2
