"""Oracle: path enumeration and the feature layouts of x, y, w and the outputs.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows "e3j ...", App. A.3 Eq. (6) (output degrees L = |l - l'| .. l + l' per pair of input
degrees), App. B.1 (parity selection rule p1 p2 = p3) and App. E.1 (trailing channels:
row = [feature coordinate][channel]).

Readings where the pages are silent:
* a path is an (x block, l2, l3) triangle with l3 <= out_lmax; its output parity is
  p3 = p1 (-1)^l2 (SH of degree l2 have parity (-1)^l2), so every triangle is kept;
* paths are ordered by (x block index, l2, l3); that order is the weight index p;
* summed mode (default): one output block per distinct (l3, p3), ordered by l3 and then
  natural parity (-1)^l3 first; paths sharing (l3, p3) add into the same block;
  per-path mode: one output block per path, in path order;
* x offsets follow the x blocks in the given order; y offsets are l2^2.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .cg import cg_block


@dataclass(frozen=True)
class Path:
    xblock: int
    l1: int
    p1: int
    l2: int
    l3: int
    p3: int
    xoff: int
    yoff: int
    out_block: int
    zoff: int


@dataclass
class Table:
    blocks: list
    sh_lmax: int
    out_lmax: int
    per_path: bool
    paths: list = field(default_factory=list)
    out_blocks: list = field(default_factory=list)   # (l3, p3)
    d1: int = 0
    d2: int = 0
    D: int = 0

    @property
    def n_paths(self) -> int:
        return len(self.paths)

    def cg(self, p: int) -> np.ndarray:
        P = self.paths[p]
        return cg_block(P.l1, P.l2, P.l3)


def make_table(blocks, sh_lmax: int, out_lmax: int, per_path: bool = False) -> Table:
    """blocks: [(l, parity)] of x in layout order."""
    xoffs, off = [], 0
    for l, _ in blocks:
        xoffs.append(off)
        off += 2 * l + 1
    d1 = off
    raw = []
    for i, (l1, p1) in enumerate(blocks):
        for l2 in range(sh_lmax + 1):
            for l3 in range(abs(l1 - l2), min(l1 + l2, out_lmax) + 1):
                raw.append((i, l1, p1, l2, l3, p1 * (-1) ** l2))
    if per_path:
        outs = [(r[4], r[5]) for r in raw]
        which = list(range(len(raw)))
    else:
        key = lambda lp: (lp[0], 0 if lp[1] == (-1) ** lp[0] else 1)
        outs = sorted({(r[4], r[5]) for r in raw}, key=key)
        which = [outs.index((r[4], r[5])) for r in raw]
    zoffs, off = [], 0
    for l3, _ in outs:
        zoffs.append(off)
        off += 2 * l3 + 1
    D = off
    paths = [Path(i, l1, p1, l2, l3, p3, xoffs[i], l2 * l2, which[k], zoffs[which[k]])
             for k, (i, l1, p1, l2, l3, p3) in enumerate(raw)]
    return Table(list(blocks), sh_lmax, out_lmax, per_path, paths, outs, d1, (sh_lmax + 1) ** 2, D)


def irreps_str(blocks, mul: int) -> str:
    return "+".join(f"{mul}x{l}{'e' if p == 1 else 'o'}" for l, p in blocks)
