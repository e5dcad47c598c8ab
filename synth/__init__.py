"""Seeded synthetic inputs shared by the oracle tests, the CUDA tests and the benchmark.

This module draws random numbers and builds neighbour graphs. It holds none of the
method's arithmetic: no spherical harmonics, no Clebsch-Gordan coefficients, no tensor
product. Everything it returns is an *input* of the method (edge vectors, node
features, edge weights, upstream gradients, a receiver-sorted CSR graph).

Seeding: every array comes from ``numpy.random.Generator(PCG64(SeedSequence(key)))`` with
``key = [workload_id, stream_id(, chunk)]``. Streams: 0 positions / unit vectors, 1 node or
row features x, 2 weights w, 3 upstream gradients (dz or dm), 4 the parameters of the radial
network that produces the weights from edge lengths. Weights and gradients are
drawn in chunks of ``CHUNK`` rows so that any subset of rows can be regenerated without
drawing the rest (the full-size parity tests sample rows that way).

Geometry follows the e3j paper's benchmark systems ("e3j: An efficient and open-source
backend for Euclidean equivariant operations on GPU and TPU", Sec. 3 and App. E.1): atoms
uniform in a periodic cubic box at 0.1 atoms/A^3, neighbours within a radial cutoff,
minimum image, no self edges, edges sorted by receiver with senders ascending inside each
receiver segment, edge vector r_ab = pos[sender] - pos[receiver].
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np

CHUNK = 4096          # rows (or edges) per independently seeded chunk
STREAM_POS, STREAM_X, STREAM_W, STREAM_GRAD, STREAM_RADIAL = 0, 1, 2, 3, 4


def rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def unit_vectors(n: int, key: tuple[int, ...]) -> np.ndarray:
    """n seeded uniform random unit 3-vectors (normalised Gaussian triples), float64."""
    g = rng(*key).standard_normal((n, 3))
    nrm = np.linalg.norm(g, axis=1, keepdims=True)
    nrm[nrm == 0] = 1.0
    return g / nrm


def _fill_chunked(out: np.ndarray, key: tuple[int, ...], scale: float, rows: np.ndarray | None):
    """Fill out[i] (i-th requested row) with N(0, scale^2) float32 draws, chunk-seeded."""
    row_shape = out.shape[1:]
    per_row = int(np.prod(row_shape)) if row_shape else 1
    flat = out.reshape(out.shape[0], per_row)
    if rows is None:
        n = out.shape[0]
        nchunks = (n + CHUNK - 1) // CHUNK

        def work(c):
            lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
            v = rng(*key, c).standard_normal((hi - lo) * per_row, dtype=np.float32)
            if scale != 1.0:
                v *= np.float32(scale)
            flat[lo:hi] = v.reshape(hi - lo, per_row)

        workers = min(16, max(1, (os.cpu_count() or 1)))
        if nchunks <= 2:
            for c in range(nchunks):
                work(c)
        else:
            with ThreadPoolExecutor(workers) as ex:
                list(ex.map(work, range(nchunks)))
    else:
        rows = np.asarray(rows, dtype=np.int64)
        chunks = np.unique(rows // CHUNK)
        for c in chunks:
            sel = np.nonzero(rows // CHUNK == c)[0]
            # regenerate the chunk up to the last requested row
            last = int(rows[sel].max() % CHUNK) + 1
            v = rng(*key, int(c)).standard_normal(last * per_row, dtype=np.float32)
            if scale != 1.0:
                v *= np.float32(scale)
            v = v.reshape(last, per_row)
            flat[sel] = v[rows[sel] % CHUNK]
    return out


def normal_rows(n_rows: int, row_shape: tuple[int, ...], key: tuple[int, ...], scale: float = 1.0,
                rows: np.ndarray | None = None) -> np.ndarray:
    """Float32 N(0, scale^2) array of shape [n_rows or len(rows), *row_shape].

    Row i of the full array is the same whether it is drawn alone (``rows=[i]``) or with all
    the others, because each chunk of CHUNK rows has its own seed.
    """
    n = n_rows if rows is None else len(rows)
    out = np.empty((n, *row_shape), dtype=np.float32)
    return _fill_chunked(out, key, scale, rows)


# ---------------------------------------------------------------------------------------
# periodic boxes and radius graphs
# ---------------------------------------------------------------------------------------

def box_side(n_atoms: int, density: float = 0.1) -> float:
    return (n_atoms / density) ** (1.0 / 3.0)


def cutoff_for_degree(k: float, density: float = 0.1) -> float:
    """Radius whose sphere holds k neighbours on average at the given density."""
    return (3.0 * k / (4.0 * math.pi * density)) ** (1.0 / 3.0)


def _morton3(ix, iy, iz):
    def spread(v):
        v = v.astype(np.uint64) & np.uint64(0x1FFFFF)
        v = (v | (v << np.uint64(32))) & np.uint64(0x1F00000000FFFF)
        v = (v | (v << np.uint64(16))) & np.uint64(0x1F0000FF0000FF)
        v = (v | (v << np.uint64(8))) & np.uint64(0x100F00F00F00F00F)
        v = (v | (v << np.uint64(4))) & np.uint64(0x10C30C30C30C30C3)
        v = (v | (v << np.uint64(2))) & np.uint64(0x1249249249249249)
        return v
    return spread(ix) | (spread(iy) << np.uint64(1)) | (spread(iz) << np.uint64(2))


@dataclass
class Graph:
    n_nodes: int
    rowptr: np.ndarray          # int32 [N+1], receiver CSR
    sender: np.ndarray          # int32 [E]
    vec: np.ndarray             # float64 [E,3], pos[sender] - pos[receiver], minimum image
    box: float = 0.0
    cutoff: float = 0.0
    order: str = "cell"
    pos: np.ndarray | None = field(default=None, repr=False)

    @property
    def n_edges(self) -> int:
        return int(self.sender.shape[0])

    def receiver(self) -> np.ndarray:
        return np.repeat(np.arange(self.n_nodes, dtype=np.int32), np.diff(self.rowptr))


def atoms_in_box(n_atoms: int, key: tuple[int, ...], density: float = 0.1, cutoff: float = 5.0,
                 order: str = "cell") -> tuple[np.ndarray, float]:
    """Uniform atoms in [0,L)^3. order='cell' renumbers atoms along a Morton curve of the
    cutoff-sized cell grid (stable inside a cell), the usual spatial sort of MD neighbour
    codes; order='draw' keeps the draw order (random)."""
    L = box_side(n_atoms, density)
    pos = rng(*key).uniform(0.0, L, size=(n_atoms, 3))
    if order == "cell":
        nc = max(1, int(L // cutoff))
        cell = np.minimum((pos / (L / nc)).astype(np.int64), nc - 1)
        code = _morton3(cell[:, 0], cell[:, 1], cell[:, 2])
        perm = np.argsort(code, kind="stable")
        pos = pos[perm]
    elif order != "draw":
        raise ValueError(order)
    return pos, L


def radius_graph(pos: np.ndarray, L: float, rc: float) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """All ordered pairs (receiver i, sender j), i != j, with minimum-image |r_j - r_i| <= rc.

    Returns (rowptr int32 [N+1], sender int32 [E], vec float64 [E,3]) sorted by receiver,
    then sender.
    """
    n = pos.shape[0]
    nc = int(L // rc)
    recv_list, send_list = [], []
    if nc < 3:
        # brute force: every pair
        for i0 in range(0, n, 1024):
            i1 = min(n, i0 + 1024)
            d = pos[None, :, :] - pos[i0:i1, None, :]
            d -= L * np.round(d / L)
            r2 = np.einsum("ijk,ijk->ij", d, d)
            ii, jj = np.nonzero(r2 <= rc * rc)
            ii = ii + i0
            keep = ii != jj
            recv_list.append(ii[keep]); send_list.append(jj[keep])
    else:
        cs = L / nc
        cidx = np.minimum((pos / cs).astype(np.int64), nc - 1)
        cid = (cidx[:, 0] * nc + cidx[:, 1]) * nc + cidx[:, 2]
        order = np.argsort(cid, kind="stable")
        counts = np.bincount(cid, minlength=nc ** 3)
        start = np.concatenate([[0], np.cumsum(counts)[:-1]])
        for dx in (-1, 0, 1):
            for dy in (-1, 0, 1):
                for dz in (-1, 0, 1):
                    nb = (((cidx[:, 0] + dx) % nc) * nc + (cidx[:, 1] + dy) % nc) * nc + (cidx[:, 2] + dz) % nc
                    cnt = counts[nb]
                    tot = int(cnt.sum())
                    if tot == 0:
                        continue
                    ii = np.repeat(np.arange(n), cnt)
                    base = np.repeat(start[nb], cnt)
                    within = np.arange(tot) - np.repeat(np.cumsum(cnt) - cnt, cnt)
                    jj = order[base + within]
                    d = pos[jj] - pos[ii]
                    d -= L * np.round(d / L)
                    r2 = np.einsum("ij,ij->i", d, d)
                    keep = (r2 <= rc * rc) & (ii != jj)
                    recv_list.append(ii[keep]); send_list.append(jj[keep])
    recv = np.concatenate(recv_list) if recv_list else np.zeros(0, np.int64)
    send = np.concatenate(send_list) if send_list else np.zeros(0, np.int64)
    srt = np.lexsort((send, recv))
    recv, send = recv[srt], send[srt]
    vec = pos[send] - pos[recv]
    vec -= L * np.round(vec / L)
    rowptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(recv, minlength=n), out=rowptr[1:])
    return rowptr.astype(np.int32), send.astype(np.int32), vec


def box_graph(workload_id: int, n_atoms: int, degree: float | None = None, cutoff: float | None = None,
              density: float = 0.1, order: str = "cell") -> Graph:
    rc = cutoff if cutoff is not None else cutoff_for_degree(degree, density)
    pos, L = atoms_in_box(n_atoms, (workload_id, STREAM_POS), density, rc, order)
    rowptr, sender, vec = radius_graph(pos, L, rc)
    return Graph(n_atoms, rowptr, sender, vec, L, rc, order, pos)


def random_graph(n_nodes: int, n_edges: int, key: tuple[int, ...], empty_nodes: int = 0) -> Graph:
    """A small irregular receiver-sorted graph for edge cases: random senders, random
    degrees (some receivers with zero edges), random edge vectors."""
    g = rng(*key)
    recv = g.integers(0, max(1, n_nodes - empty_nodes), size=n_edges) if n_edges else np.zeros(0, np.int64)
    send = g.integers(0, n_nodes, size=n_edges) if n_edges else np.zeros(0, np.int64)
    srt = np.lexsort((send, recv))
    recv, send = recv[srt], send[srt]
    rowptr = np.zeros(n_nodes + 1, dtype=np.int64)
    np.cumsum(np.bincount(recv, minlength=n_nodes), out=rowptr[1:])
    vec = g.standard_normal((n_edges, 3))
    return Graph(n_nodes, rowptr.astype(np.int32), send.astype(np.int32), vec, 0.0, 0.0, "random")


def padded_graph(g: Graph, n_self: int, n_out: int, n_in: int, key: tuple[int, ...]):
    """g plus one padding node (index g.n_nodes) and padding edges, the static-shape layout of
    JAX graph codes (e3j, Sec. 4 "Message passing convolution": unused edge slots all point at
    one padding node). n_self edges pad -> pad, n_out edges pad -> a random real receiver,
    n_in edges a random real sender -> pad. Padding edges are placed at random positions
    inside their receiver's segment; real edges keep their relative order. Returns
    (graph, pad, orig): orig[e] is the index in g of new edge e, or -1 for padding edges.
    Padding edge vectors are NaN."""
    r = rng(*key)
    N, pad = g.n_nodes, g.n_nodes
    recv0 = g.receiver().astype(np.int64)
    deg = np.diff(g.rowptr.astype(np.int64))
    rank = np.arange(g.n_edges) - np.repeat(g.rowptr[:-1].astype(np.int64), deg)
    p_recv = np.concatenate([np.full(n_self, pad), r.integers(0, N, n_out), np.full(n_in, pad)]).astype(np.int64)
    p_send = np.concatenate([np.full(n_self, pad), np.full(n_out, pad), r.integers(0, N, n_in)]).astype(np.int64)
    degp = np.concatenate([deg, [0]])
    p_posn = r.uniform(-0.5, degp[p_recv] + 0.5)
    recv = np.concatenate([recv0, p_recv])
    send = np.concatenate([g.sender.astype(np.int64), p_send])
    posn = np.concatenate([rank.astype(np.float64), p_posn])
    orig = np.concatenate([np.arange(g.n_edges), np.full(len(p_recv), -1)])
    srt = np.lexsort((posn, recv))
    recv, send, orig = recv[srt], send[srt], orig[srt]
    rowptr = np.zeros(N + 2, dtype=np.int64)
    np.cumsum(np.bincount(recv, minlength=N + 1), out=rowptr[1:])
    vec = np.full((len(orig), 3), np.nan)
    vec[orig >= 0] = g.vec[orig[orig >= 0]]
    out = Graph(N + 1, rowptr.astype(np.int32), send.astype(np.int32), vec, g.box, g.cutoff, g.order + "+pad")
    return out, pad, orig


def device_normal(shape: tuple[int, ...], key: tuple[int, ...], scale: float = 1.0, device="cuda",
                  dtype=None):
    """Seeded N(0, scale^2) float32 tensor drawn on the GPU with torch's generator (for inputs
    of tens of GB, e.g. the per-edge weights of the 64k-atom workload). The seed is derived
    from key like the host streams; both sides of a comparison read the same tensor (the
    oracle copies the rows it samples to the host)."""
    import torch
    seed = int(np.random.SeedSequence([int(k) for k in key]).generate_state(1, np.uint64)[0] >> np.uint64(1))
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    if dtype is not None and dtype != torch.float32:
        t = t.to(dtype)
    return t
