"""The oracle: a plain, slow, float64 CPU statement of what the hot path computes.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package. The product (the CUDA library in
``message_passing_gb300``) never imports, links or runs anything here, and this package
shares no code with it: its own SH polynomials (sh.py), its own CG construction (cg.py,
null space of the equivariance constraint), its own path enumeration (paths.py) and plain
C loops (tp.c) for the tensor product and convolution.

Pins (tests/test_oracle_*.py, marker ``not gpu``) tie every function to facts outside the
oracle: closed forms of the harmonics, the addition theorem, harmonicity and parity;
orthogonality and closed forms (dot, cross, identity) of the CG blocks and equivariance
under rotations whose Wigner matrices are fitted from harmonic values; equivariance of the
tensor product and convolution, a scalar-only case that is a plain weighted SpMM, the
Euler identity <dz, z> = <dx, x> = <dy, y> = <dw, w> and central finite differences for the
backward passes, and the convolution as a scatter-sum (numpy.add.at) of per-edge products.
The radial edge scalars (radial.py: Bessel basis, polynomial envelope, one SiLU hidden layer)
are pinned by scipy's spherical Bessel functions, quadrature, the envelope's defining
conditions, finite differences and the forces of the radial-weighted convolution.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .cg import cg_block
from .coo import cg_records, coo_tp_backward, coo_tp_forward
from . import radial
from .paths import Table, make_table
from .sh import sh, sh_grad

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile tp.c with gcc (OpenMP when available). No FMA contraction, so x86 and Arm
    give the same bits."""
    src = os.path.join(_HERE, "tp.c")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(src):
        return _LIB
    os.makedirs(_LIBDIR, exist_ok=True)
    tmp = _LIB + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", src, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.orc_tp_forward.argtypes = [i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.orc_tp_backward.argtypes = [i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                            vp, vp, vp]
            lib.orc_conv_forward.argtypes = [i64, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                             vp, dbl, vp]
            lib.orc_conv_backward_edges.argtypes = [i64, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                                    vp, vp, vp, vp, dbl, vp, vp]
            lib.orc_conv_backward_dx.argtypes = [i64, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                                 vp, vp, dbl, vp]
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def table(blocks, sh_lmax: int, out_lmax: int, per_path: bool = False) -> Table:
    return make_table(blocks, sh_lmax, out_lmax, per_path)


def _pack(t: Table):
    pinfo = np.zeros((t.n_paths, 7), dtype=np.int32)
    blocks, off = [], 0
    for k, p in enumerate(t.paths):
        C = cg_block(p.l1, p.l2, p.l3)
        pinfo[k] = (p.xoff, p.yoff, p.zoff, 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1, off)
        blocks.append(C.reshape(-1))
        off += C.size
    cg = np.ascontiguousarray(np.concatenate(blocks) if blocks else np.zeros(1))
    return np.ascontiguousarray(pinfo), cg


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def tp_forward(t: Table, x, y, w):
    """z[R, D, Nq] (Eq. 10-11)."""
    x, y, w = _f64(x), _f64(y), _f64(w)
    R, d1, Nq = x.shape
    assert d1 == t.d1 and y.shape == (R, t.d2) and w.shape == (R, t.n_paths, Nq)
    pinfo, cg = _pack(t)
    z = np.empty((R, t.D, Nq))
    _load().orc_tp_forward(R, t.d1, t.d2, t.D, t.n_paths, Nq, _p(pinfo), _p(cg), _p(x), _p(y),
                           _p(w), _p(z))
    return z


def tp_backward(t: Table, x, y, w, dz):
    """(dx, dy, dw) (Eq. 15, with the per-path weights as a third operand)."""
    x, y, w, dz = _f64(x), _f64(y), _f64(w), _f64(dz)
    R, d1, Nq = x.shape
    assert dz.shape == (R, t.D, Nq)
    pinfo, cg = _pack(t)
    dx = np.empty_like(x)
    dy = np.empty((R, t.d2))
    dw = np.empty_like(w)
    _load().orc_tp_backward(R, t.d1, t.d2, t.D, t.n_paths, Nq, _p(pinfo), _p(cg), _p(x), _p(y),
                            _p(w), _p(dz), _p(dx), _p(dy), _p(dw))
    return dx, dy, dw


def _segments(ptr, ids):
    ids = np.asarray(ids, dtype=np.int64)
    lo = ptr[ids].astype(np.int64)
    hi = ptr[ids + 1].astype(np.int64)
    cnt = hi - lo
    sub = np.zeros(len(ids) + 1, dtype=np.int64)
    np.cumsum(cnt, out=sub[1:])
    edges = np.repeat(lo - sub[:-1], cnt) + np.arange(int(sub[-1]), dtype=np.int64)
    return sub, edges


def _drop_padding(sub, edges, owner, other, pad):
    """Remove the padding edges from per-node edge lists (sub offsets, edges ids): an edge is
    padding when its owning node (owner[i] for list position i) or its other end (other[i])
    is the padding node. e3j, Sec. 4 "Message passing convolution" and App. E: static-shape
    graphs send their unused edge slots to one padding node, and the kernels skip them."""
    if pad is None or pad < 0:
        return sub, edges
    keep = (owner != pad) & (other != pad)
    seg = np.repeat(np.arange(len(sub) - 1), np.diff(sub))      # list position -> node slot
    kept = np.zeros(len(sub), dtype=np.int64)
    np.cumsum(np.bincount(seg[keep], minlength=len(sub) - 1), out=kept[1:])
    return kept, edges[keep]


def conv_forward(t: Table, rowptr, sender, x, y, w, scale: float, receivers=None, pad_node=None):
    """m[len(receivers), D, Nq] = scale * sum over each receiver's CSR edges (Eq. 12-13).
    y and w are per-edge arrays over all edges (or callables edge_ids -> rows). With pad_node,
    the edges whose receiver or sender is pad_node contribute nothing."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    n = rowptr.shape[0] - 1
    recv = np.arange(n) if receivers is None else np.asarray(receivers, dtype=np.int64)
    sub, edges = _segments(rowptr, recv)
    sub, edges = _drop_padding(sub, edges, np.repeat(recv, np.diff(sub)), np.asarray(sender)[edges], pad_node)
    snd = np.ascontiguousarray(np.asarray(sender)[edges], dtype=np.int32)
    ye = _f64(y(edges) if callable(y) else np.asarray(y)[edges])
    we = _f64(w(edges) if callable(w) else np.asarray(w)[edges])
    x = _f64(x)
    Nq = x.shape[2]
    pinfo, cg = _pack(t)
    m = np.empty((len(recv), t.D, Nq))
    _load().orc_conv_forward(len(recv), _p(sub), _p(snd), t.d1, t.d2, t.D, t.n_paths, Nq,
                             _p(pinfo), _p(cg), _p(x), _p(ye), _p(we), float(scale), _p(m))
    return m


def receivers_of(rowptr) -> np.ndarray:
    rowptr = np.asarray(rowptr, dtype=np.int64)
    return np.repeat(np.arange(rowptr.shape[0] - 1, dtype=np.int32), np.diff(rowptr))


def conv_backward_edges(t: Table, rowptr, sender, x, y, w, dm, scale: float, edges=None, pad_node=None):
    """(dy[len(edges), d2], dw[len(edges), P, Nq]) for the given edge ids (Eq. 16). A padding
    edge (receiver or sender == pad_node) takes no part in the forward, so both are zero."""
    sender = np.asarray(sender)
    E = sender.shape[0]
    edges = np.arange(E) if edges is None else np.asarray(edges, dtype=np.int64)
    if pad_node is not None and pad_node >= 0:
        rcv = receivers_of(rowptr)[edges]
        real = (rcv != pad_node) & (sender[edges] != pad_node)
        Nq = np.asarray(x).shape[2]
        dy = np.zeros((len(edges), t.d2))
        dw = np.zeros((len(edges), t.n_paths, Nq))
        if real.any():
            dy[real], dw[real] = conv_backward_edges(t, rowptr, sender, x, y, w, dm, scale, edges[real])
        return dy, dw
    recv = receivers_of(rowptr)[edges]
    snd = np.ascontiguousarray(sender[edges], dtype=np.int32)
    ye = _f64(y(edges) if callable(y) else np.asarray(y)[edges])
    we = _f64(w(edges) if callable(w) else np.asarray(w)[edges])
    x, dm = _f64(x), _f64(dm)
    Nq = x.shape[2]
    pinfo, cg = _pack(t)
    dy = np.empty((len(edges), t.d2))
    dw = np.empty((len(edges), t.n_paths, Nq))
    _load().orc_conv_backward_edges(len(edges), _p(snd), _p(np.ascontiguousarray(recv, np.int32)),
                                    t.d1, t.d2, t.D, t.n_paths, Nq, _p(pinfo), _p(cg), _p(x),
                                    _p(ye), _p(we), _p(dm), float(scale), _p(dy), _p(dw))
    return dy, dw


def conv_backward_dx(t: Table, rowptr, sender, y, w, dm, scale: float, senders=None, Nq=None, pad_node=None):
    """dx[len(senders), d1, Nq]: sum over the edges whose sender is each node (Eq. 16); with
    pad_node, over the edges that are not padding (receiver and sender != pad_node)."""
    sender = np.asarray(sender, dtype=np.int64)
    n = np.asarray(rowptr).shape[0] - 1
    dm = _f64(dm)
    Nq = dm.shape[2] if Nq is None else Nq
    nodes = np.arange(n) if senders is None else np.asarray(senders, dtype=np.int64)
    recv_all = receivers_of(rowptr)
    # edges of each requested sender, in edge order
    order = np.argsort(sender, kind="stable")
    cptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(sender, minlength=n), out=cptr[1:])
    sub, pos = _segments(cptr, nodes)
    edges = order[pos]
    sub, edges = _drop_padding(sub, edges, np.repeat(nodes, np.diff(sub)), recv_all[edges], pad_node)
    ye = _f64(y(edges) if callable(y) else np.asarray(y)[edges])
    we = _f64(w(edges) if callable(w) else np.asarray(w)[edges])
    pinfo, cg = _pack(t)
    dx = np.empty((len(nodes), t.d1, Nq))
    _load().orc_conv_backward_dx(len(nodes), _p(sub),
                                 _p(np.ascontiguousarray(recv_all[edges], np.int32)), t.d1, t.d2,
                                 t.D, t.n_paths, Nq, _p(pinfo), _p(cg), _p(ye), _p(we), _p(dm),
                                 float(scale), _p(dx))
    return dx


def conv_double_backward(t: Table, rowptr, sender, x, y, w, dm, ddx, ddy, ddw, scale: float,
                         receivers=None, senders=None, edges=None, pad_node=None):
    """Second-order rule of the convolution, e3j App. E.1 Eq. (17)-(18): with (ddx, ddy, ddw)
    the variations of the cotangents (dx, dy, dw) returned by the backward pass,

      delta dm = conv(ddx, y, w) + conv(x, ddy, w) + conv(x, y, ddw)                     (17)
      (-, dx_y, dx_w) = conv_bwd(ddx, y, w, dm)                                          (18)
      (dy_x, -, dy_w) = conv_bwd(x, ddy, w, dm)
      (dw_x, dw_y, -) = conv_bwd(x, y, ddw, dm)
      delta x = dy_x + dw_x,  delta y = dx_y + dw_y,  delta w = dx_w + dy_w

    (the table's labels: each conv_bwd call returns (dx, dy, dw) of its own arguments).
    Returns (delta_x[senders], delta_y[edges], delta_w[edges], delta_dm[receivers]).
    y, w, ddy, ddw may be callables edge_ids -> rows."""
    sender = np.asarray(sender)
    n = np.asarray(rowptr).shape[0] - 1
    Nq = np.asarray(x).shape[2]
    kw = dict(pad_node=pad_node)
    # (17)
    ddm = (conv_forward(t, rowptr, sender, ddx, y, w, scale, receivers, **kw)
           + conv_forward(t, rowptr, sender, x, ddy, w, scale, receivers, **kw)
           + conv_forward(t, rowptr, sender, x, y, ddw, scale, receivers, **kw))
    # (18): the three conv_bwd calls, each with one primal replaced by its variation
    dy1, dw1 = conv_backward_edges(t, rowptr, sender, ddx, y, w, dm, scale, edges, **kw)
    dx2 = conv_backward_dx(t, rowptr, sender, ddy, w, dm, scale, senders, Nq, **kw)
    _, dw2 = conv_backward_edges(t, rowptr, sender, x, ddy, w, dm, scale, edges, **kw)
    dx3 = conv_backward_dx(t, rowptr, sender, y, ddw, dm, scale, senders, Nq, **kw)
    dy3, _ = conv_backward_edges(t, rowptr, sender, x, y, ddw, dm, scale, edges, **kw)
    return dx2 + dx3, dy1 + dy3, dw1 + dw2, ddm


__all__ = ["radial", "sh", "sh_grad", "cg_block", "cg_records", "coo_tp_forward", "coo_tp_backward", "table", "tp_forward",
           "tp_backward", "conv_forward",
           "conv_backward_edges", "conv_backward_dx", "conv_double_backward", "build", "num_threads",
           "receivers_of"]
