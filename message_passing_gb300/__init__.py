"""Python binding of libe3gb.so (include/e3gb.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; PyTorch provides device
memory and streams. The functions keep the C names without the ``e3gb_`` prefix and take
torch tensors. If the library is missing or fails to load, importing the functions raises
(there is no CPU path).

Operations follow "e3j: An efficient and open-source backend for Euclidean equivariant
operations on GPU and TPU", App. E.1 Eq. (10)-(16); see include/e3gb.h for layouts.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libe3gb.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_BAD_GRAPH, ERR_DEVICE_INDEX = range(6)
F32, BF16 = 0, 1
PATHS_SUMMED, PATHS_SEPARATE = 0, 1

# every symbol include/e3gb.h declares
SYMBOLS = (
    "e3gb_table_create", "e3gb_table_destroy", "e3gb_table_info", "e3gb_table_paths",
    "e3gb_table_coefficients", "e3gb_config_count", "e3gb_config_describe", "e3gb_sh_forward",
    "e3gb_sh_backward",
    "e3gb_tp_forward", "e3gb_tp_backward", "e3gb_graph_prepare_workspace_bytes",
    "e3gb_graph_prepare", "e3gb_graph_prepare_static", "e3gb_conv_forward", "e3gb_conv_backward",
    "e3gb_conv_double_backward", "e3gb_coo_tp_forward", "e3gb_coo_tp_backward",
    "e3gb_radial_hidden", "e3gb_radial_backward", "e3gb_conv_forward_radial", "e3gb_conv_backward_radial",
    "e3gb_conv_forward_split_workspace_bytes", "e3gb_conv_forward_split",
    "e3gb_check_device_status", "e3gb_last_error", "e3gb_version",
)

# hidden width the radial convolution kernels are built for
RADIAL_HIDDEN = 8


class E3GBError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"e3gb status {status}: {msg}")
        self.status = status


class _Irreps(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("l", ctypes.POINTER(ctypes.c_int32)),
                ("parity", ctypes.POINTER(ctypes.c_int32)), ("mul", ctypes.c_int32)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libe3gb.so (built by message_passing_gb300.build). Raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with message_passing_gb300.build.build()")
    lib = ctypes.CDLL(p)
    i32, i64, vp, f32, szt = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
    P32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "e3gb_table_create": (i32, [ctypes.POINTER(_Irreps), i32, i32, i32, ctypes.POINTER(vp)]),
        "e3gb_table_destroy": (i32, [vp]),
        "e3gb_table_info": (i32, [vp, P32, P32, P32, P32, P32, P32]),
        "e3gb_table_paths": (i32, [vp, P32]),
        "e3gb_table_coefficients": (i32, [vp, ctypes.POINTER(ctypes.c_double)]),
        "e3gb_config_count": (i32, []),
        "e3gb_config_describe": (i32, [i32, P32, P32, P32, P32, P32, P32]),
        "e3gb_sh_forward": (i32, [i32, i64, vp, vp, i32, vp]),
        "e3gb_sh_backward": (i32, [i32, i64, vp, vp, vp, i32, vp]),
        "e3gb_tp_forward": (i32, [vp, i64, vp, vp, vp, vp, i32, vp]),
        "e3gb_tp_backward": (i32, [vp, i64, vp, vp, vp, vp, vp, vp, vp, i32, vp]),
        "e3gb_graph_prepare_workspace_bytes": (szt, [i64, i64]),
        "e3gb_graph_prepare": (i32, [i64, i64, vp, vp, vp, vp, vp, vp, szt, vp]),
        "e3gb_graph_prepare_static": (i32, [i64, i64, vp, vp, vp, vp, vp, vp]),
        "e3gb_conv_forward": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, f32, i64, vp, i32, vp]),
        "e3gb_conv_backward": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, f32, i64, vp, vp, vp, i32, vp]),
        "e3gb_conv_double_backward": (i32, [vp, i64, i64] + [vp] * 5 + [vp] * 7 + [f32, i64] + [vp] * 4
                                      + [i32, vp]),
        "e3gb_coo_tp_forward": (i32, [i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp]),
        "e3gb_coo_tp_backward": (i32, [i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                       vp]),
        "e3gb_radial_hidden": (i32, [i64, vp, vp, i32, i32, f32, vp, vp]),
        "e3gb_radial_backward": (i32, [i64, vp, vp, i32, i32, f32, vp, vp, i32, vp]),
        "e3gb_conv_forward_radial": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, vp, i32, f32, i64, vp, i32, vp]),
        "e3gb_conv_backward_radial": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, i32, vp, f32, i64, vp, vp, vp,
                                            i32, vp]),
        "e3gb_conv_forward_split_workspace_bytes": (szt, [vp, i64, i64, i32]),
        "e3gb_conv_forward_split": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, f32, i64, i32, vp, vp, szt, i32, vp]),
        "e3gb_check_device_status": (i32, [vp, P32]),
        "e3gb_last_error": (ctypes.c_char_p, []),
        "e3gb_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        raise E3GBError(status, load().e3gb_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(*ts):
    import torch
    dt = {t.dtype for t in ts if t is not None}
    if dt == {torch.float32}:
        return F32
    if dt == {torch.bfloat16}:
        return BF16
    raise TypeError(f"tensors must all be float32 or all bfloat16, got {dt}")


def _f32_out(*ts):
    import torch
    for t in ts:
        if t is not None and t.dtype != torch.float32:
            raise TypeError("outputs are float32 in both the fp32 and the bf16 variant")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _shape(name, t, *shape):
    """The kernels index every buffer from the table's sizes and the row/node/edge counts, so a
    buffer of another shape would be read or written out of bounds: refuse it here."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _index_len(name, t, n):
    """An index array of at least n entries (the graph index arrays hold max(E, 1))."""
    if t is not None and (t.dim() != 1 or t.shape[0] < n):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected ({n},) or longer")


def version() -> str:
    return load().e3gb_version().decode()


def configs() -> list[dict]:
    """The irreps configurations compiled into the library."""
    lib = load()
    out = []
    for i in range(lib.e3gb_config_count()):
        n = ctypes.c_int32()
        l = (ctypes.c_int32 * 8)()
        p = (ctypes.c_int32 * 8)()
        a, b, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib.e3gb_config_describe(i, ctypes.byref(n), l, p, ctypes.byref(a), ctypes.byref(b), ctypes.byref(f)))
        out.append({"blocks": [(l[k], p[k]) for k in range(n.value)], "sh_lmax": a.value,
                    "out_lmax": b.value, "per_path": bool(f.value)})
    return out


@dataclass
class Table:
    """Path table handle (e3gb_table). blocks: [(l, parity)] of x; mul: channels."""
    handle: ctypes.c_void_p
    blocks: list
    mul: int
    sh_lmax: int
    out_lmax: int
    per_path: bool
    d1: int = 0
    d2: int = 0
    n_paths: int = 0
    D: int = 0
    nnz: int = 0

    @classmethod
    def create(cls, blocks, mul: int, sh_lmax: int, out_lmax: int, per_path: bool = False) -> "Table":
        lib = load()
        n = len(blocks)
        L = (ctypes.c_int32 * max(1, n))(*[b[0] for b in blocks])
        P = (ctypes.c_int32 * max(1, n))(*[b[1] for b in blocks])
        ir = _Irreps(n, L, P, mul)
        h = ctypes.c_void_p()
        _check(lib.e3gb_table_create(ctypes.byref(ir), sh_lmax, out_lmax,
                                     PATHS_SEPARATE if per_path else PATHS_SUMMED, ctypes.byref(h)))
        t = cls(h, list(blocks), mul, sh_lmax, out_lmax, per_path)
        v = [ctypes.c_int32() for _ in range(6)]
        _check(lib.e3gb_table_info(h, *[ctypes.byref(x) for x in v]))
        t.d1, t.d2, t.n_paths, t.D, t.nnz, _ = (x.value for x in v)
        return t

    def paths(self) -> list[tuple]:
        buf = (ctypes.c_int32 * (8 * self.n_paths))()
        _check(load().e3gb_table_paths(self.handle, buf))
        return [tuple(buf[8 * i:8 * i + 8]) for i in range(self.n_paths)]

    def coefficients(self):
        import numpy as np
        buf = (ctypes.c_double * (5 * self.nnz))()
        _check(load().e3gb_table_coefficients(self.handle, buf))
        return np.frombuffer(buf, dtype=np.float64).reshape(self.nnz, 5).copy()

    def coo_records(self):
        """The table's CG tensor product as records for coo_tp_forward: (int32 [n,4] rows
        (i0, i1, i2, path), float32 [n] coefficients), host arrays."""
        import numpy as np
        xoff = np.concatenate([[0], np.cumsum([2 * l + 1 for l, _ in self.blocks])])
        paths = np.array(self.paths(), dtype=np.int64).reshape(-1, 8)
        co = self.coefficients()
        p = co[:, 0].astype(np.int64)
        rec = np.stack([paths[p, 7] + co[:, 3].astype(np.int64),            # output offset + m3
                        xoff[paths[p, 0]] + co[:, 1].astype(np.int64),      # x block offset + m1
                        paths[p, 3] ** 2 + co[:, 2].astype(np.int64),       # l2^2 + m2
                        p], axis=1).astype(np.int32)
        return np.ascontiguousarray(rec), co[:, 4].astype(np.float32)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.e3gb_table_destroy(h)
            self.handle = None


def _rows_operands(t: "Table", R: int, x, y, w, names=("x", "y", "w")):
    _shape(names[0], x, R, t.d1, t.mul)
    _shape(names[1], y, R, t.d2)
    _shape(names[2], w, R, t.n_paths, t.mul)


def _conv_operands(t: "Table", N: int, E: int, x, y, w, names=("x", "y", "w")):
    _shape(names[0], x, N, t.d1, t.mul)
    _shape(names[1], y, E, t.d2)
    _shape(names[2], w, E, t.n_paths, t.mul)


def _csc_shapes(csc, N: int, E: int):
    cp, ce, cr = csc
    _shape("csc_ptr", cp, N + 1)
    _index_len("csc_edge", ce, E)
    _index_len("csc_recv", cr, E)


def sh_forward(vec, lmax: int, out=None, dtype=None, stream=None):
    """y[n, (lmax+1)^2] = real SH of vec[n, 3] (fp32 device tensor)."""
    import torch
    _contig(vec)
    if vec.dtype != torch.float32:
        raise TypeError("vec must be float32")
    dt = dtype or torch.float32
    _shape("vec", vec, vec.shape[0], 3)
    y = out if out is not None else torch.empty((vec.shape[0], (lmax + 1) ** 2), dtype=dt, device=vec.device)
    _shape("y", y, vec.shape[0], (lmax + 1) ** 2)
    _check(load().e3gb_sh_forward(lmax, vec.shape[0], _ptr(vec), _ptr(y), _dtype(y), _stream(stream)))
    return y


def sh_backward(vec, dy, lmax: int, out=None, stream=None):
    """dvec[n, 3] (fp32) = VJP of sh_forward for the cotangent dy[n, (lmax+1)^2]."""
    import torch
    _contig(vec, dy)
    if vec.dtype != torch.float32:
        raise TypeError("vec must be float32")
    n = vec.shape[0]
    _shape("vec", vec, n, 3)
    _shape("dy", dy, n, (lmax + 1) ** 2)
    dvec = out if out is not None else torch.empty((n, 3), dtype=torch.float32, device=vec.device)
    _shape("dvec", dvec, n, 3)
    _f32_out(dvec)
    _check(load().e3gb_sh_backward(lmax, vec.shape[0], _ptr(vec), _ptr(dy), _ptr(dvec), _dtype(dy), _stream(stream)))
    return dvec


def tp_forward(t: Table, x, y, w, out=None, stream=None):
    """z[R, D, mul] (fp32) = sum over paths of w * CG(x, y) per row: x [R, d1, mul],
    y [R, d2], w [R, n_paths, mul]."""
    import torch
    _contig(x, y, w, out)
    R = x.shape[0]
    _rows_operands(t, R, x, y, w)
    z = out if out is not None else torch.empty((R, t.D, t.mul), dtype=torch.float32, device=x.device)
    _shape("z", z, R, t.D, t.mul)
    _f32_out(z)
    _check(load().e3gb_tp_forward(t.handle, x.shape[0], _ptr(x), _ptr(y), _ptr(w), _ptr(z),
                                  _dtype(x, y, w), _stream(stream)))
    return z


def tp_backward(t: Table, x, y, w, dz, out=None, stream=None):
    """(dx, dy, dw) of tp_forward for the cotangent dz [R, D, mul], all fp32, shaped like
    x, y, w."""
    import torch
    _contig(x, y, w, dz)
    R = x.shape[0]
    _rows_operands(t, R, x, y, w)
    _shape("dz", dz, R, t.D, t.mul)
    if out is None:
        f = dict(dtype=torch.float32)
        out = (torch.empty_like(x, **f), torch.empty_like(y, **f), torch.empty_like(w, **f))
    dx, dy, dw = out
    _rows_operands(t, R, dx, dy, dw, ("dx", "dy", "dw"))
    _f32_out(dx, dy, dw)
    _check(load().e3gb_tp_backward(t.handle, x.shape[0], _ptr(x), _ptr(y), _ptr(w), _ptr(dz), _ptr(dx),
                                   _ptr(dy), _ptr(dw), _dtype(x, y, w, dz), _stream(stream)))
    return dx, dy, dw


def graph_prepare_workspace_bytes(n_nodes: int, n_edges: int) -> int:
    return int(load().e3gb_graph_prepare_workspace_bytes(n_nodes, n_edges))


def graph_prepare(rowptr, sender, n_nodes: int, out=None, workspace=None, stream=None):
    """(csc_ptr, csc_edge, csc_recv) int32 device tensors."""
    import torch
    _contig(rowptr, sender)
    E = sender.shape[0]
    dev = rowptr.device
    _shape("rowptr", rowptr, n_nodes + 1)
    if out is None:
        out = (torch.empty(n_nodes + 1, dtype=torch.int32, device=dev),
               torch.empty(max(E, 1), dtype=torch.int32, device=dev),
               torch.empty(max(E, 1), dtype=torch.int32, device=dev))
    _csc_shapes(out, n_nodes, E)
    nb = graph_prepare_workspace_bytes(n_nodes, E)
    ws = workspace if workspace is not None else torch.empty(nb, dtype=torch.uint8, device=dev)
    cp, ce, cr = out
    _check(load().e3gb_graph_prepare(n_nodes, E, _ptr(rowptr), _ptr(sender) if E else None, _ptr(cp),
                                     _ptr(ce) if E else None, _ptr(cr) if E else None, _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))
    return cp, ce, cr


STATIC_PREPARE_SCRATCH_BYTES = 4 << 20


def graph_prepare_static(rowptr, sender, n_nodes: int, out=None, stream=None):
    """graph_prepare without a workspace, for callers that cannot allocate device memory:
    the library keeps the sort's digit counts in its own static device array of
    STATIC_PREPARE_SCRATCH_BYTES (calls overlapping on the GPU race on it). Pass ``out``
    to avoid allocating the outputs here too."""
    import torch
    _contig(rowptr, sender)
    E = sender.shape[0]
    dev = rowptr.device
    _shape("rowptr", rowptr, n_nodes + 1)
    if out is None:
        out = (torch.empty(n_nodes + 1, dtype=torch.int32, device=dev),
               torch.empty(max(E, 1), dtype=torch.int32, device=dev),
               torch.empty(max(E, 1), dtype=torch.int32, device=dev))
    _csc_shapes(out, n_nodes, E)
    cp, ce, cr = out
    _check(load().e3gb_graph_prepare_static(n_nodes, E, _ptr(rowptr), _ptr(sender) if E else None, _ptr(cp),
                                            _ptr(ce) if E else None, _ptr(cr) if E else None, _stream(stream)))
    return cp, ce, cr


def conv_forward(t: Table, rowptr, sender, x, y, w, scale: float, out=None, stream=None, pad_node: int = -1):
    """m = scale * sum over each receiver's CSR edges of TP(x[sender], y, w); edges touching
    pad_node (>= 0) are padding and skipped."""
    import torch
    _contig(rowptr, sender, x, y, w)
    N, E = x.shape[0], sender.shape[0]
    _shape("rowptr", rowptr, N + 1)
    _conv_operands(t, N, E, x, y, w)
    m = out if out is not None else torch.empty((N, t.D, t.mul), dtype=torch.float32, device=x.device)
    _shape("m", m, N, t.D, t.mul)
    _f32_out(m)
    _check(load().e3gb_conv_forward(t.handle, N, E, _ptr(rowptr), _ptr(sender) if E else None, _ptr(x),
                                    _ptr(y) if E else None, _ptr(w) if E else None, float(scale), int(pad_node), _ptr(m),
                                    _dtype(x, *((y, w) if E else ())), _stream(stream)))
    return m


def conv_forward_split(t: Table, rowptr, sender, x, y, w, scale: float, chunk: int = 256, out=None, workspace=None,
                       stream=None, pad_node: int = -1):
    """conv_forward with receivers of more than `chunk` edges cut into pieces summed by separate
    warps and added in piece order (deterministic); for graphs with heavy receivers."""
    import torch
    _contig(rowptr, sender, x, y, w)
    N, E = x.shape[0], sender.shape[0]
    _shape("rowptr", rowptr, N + 1)
    _conv_operands(t, N, E, x, y, w)
    m = out if out is not None else torch.empty((N, t.D, t.mul), dtype=torch.float32, device=x.device)
    _shape("m", m, N, t.D, t.mul)
    _f32_out(m)
    nb = int(load().e3gb_conv_forward_split_workspace_bytes(t.handle, N, E, int(chunk)))
    ws = workspace if workspace is not None else torch.empty(max(nb, 16), dtype=torch.uint8, device=x.device)
    _check(load().e3gb_conv_forward_split(t.handle, N, E, _ptr(rowptr), _ptr(sender) if E else None, _ptr(x),
                                          _ptr(y) if E else None, _ptr(w) if E else None, float(scale), int(pad_node),
                                          int(chunk), _ptr(m), _ptr(ws), ws.numel() * ws.element_size(),
                                          _dtype(x, *((y, w) if E else ())), _stream(stream)))
    return m


def conv_backward(t: Table, csc, x, y, w, dm, scale: float, out=None, stream=None, pad_node: int = -1):
    """csc = graph_prepare(...) output. Returns (dx, dy, dw); padding edges (touching
    pad_node >= 0) get zero dy and dw rows."""
    import torch
    cp, ce, cr = csc
    _contig(x, y, w, dm)
    N, E = x.shape[0], y.shape[0]
    _csc_shapes(csc, N, E)
    _conv_operands(t, N, E, x, y, w)
    _shape("dm", dm, N, t.D, t.mul)
    if out is None:
        f = dict(dtype=torch.float32)
        out = (torch.empty_like(x, **f), torch.empty_like(y, **f), torch.empty_like(w, **f))
    dx, dy, dw = out
    _conv_operands(t, N, E, dx, dy, dw, ("dx", "dy", "dw"))
    _f32_out(dx, dy, dw)
    _check(load().e3gb_conv_backward(t.handle, N, E, _ptr(cp), _ptr(ce) if E else None, _ptr(cr) if E else None,
                                     _ptr(x), _ptr(y) if E else None, _ptr(w) if E else None, _ptr(dm),
                                     float(scale), int(pad_node), _ptr(dx), _ptr(dy) if E else None,
                                     _ptr(dw) if E else None,
                                     _dtype(x, dm, *((y, w) if E else ())), _stream(stream)))
    return dx, dy, dw


def radial_hidden(vec, W1, r_cut: float, out=None, stream=None):
    """h [E, hidden] = silu(bessel_basis(|vec|) @ W1): the hidden layer of the radial network
    (W1 [n_basis, hidden], fp32 device tensors)."""
    import torch
    _contig(vec, W1)
    E = vec.shape[0]
    _shape("vec", vec, E, 3)
    nb, H = W1.shape
    h = out if out is not None else torch.empty((E, H), dtype=torch.float32, device=vec.device)
    _shape("h", h, E, H)
    for n, a in (("vec", vec), ("W1", W1), ("h", h)):
        if a.dtype != torch.float32:
            raise TypeError(f"{n} must be float32")
    _check(load().e3gb_radial_hidden(E, _ptr(vec) if E else None, _ptr(W1), nb, H, float(r_cut),
                                     _ptr(h) if E else None, _stream(stream)))
    return h


def radial_backward(vec, W1, r_cut: float, dh, out=None, accumulate: bool = False, stream=None):
    """dvec [E, 3] = d<dh, h>/dvec (forces through the radial weights); accumulate adds to out."""
    import torch
    _contig(vec, W1, dh)
    E = vec.shape[0]
    nb, H = W1.shape
    _shape("vec", vec, E, 3)
    _shape("dh", dh, E, H)
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs out")
        out = torch.empty((E, 3), dtype=torch.float32, device=vec.device)
    _shape("dvec", out, E, 3)
    _check(load().e3gb_radial_backward(E, _ptr(vec) if E else None, _ptr(W1), nb, H, float(r_cut),
                                       _ptr(dh) if E else None, _ptr(out) if E else None, int(bool(accumulate)),
                                       _stream(stream)))
    return out


def _radial_operands(t: "Table", E: int, h, W2):
    _shape("h", h, E, RADIAL_HIDDEN)
    _shape("W2", W2, RADIAL_HIDDEN, t.n_paths, t.mul)


def conv_forward_radial(t: Table, rowptr, sender, x, y, h, W2, scale: float, out=None, stream=None,
                        pad_node: int = -1):
    """conv_forward with w[e] = h[e] @ W2 formed inside the kernel (never stored); fp32."""
    import torch
    _contig(rowptr, sender, x, y, h, W2)
    N, E = x.shape[0], sender.shape[0]
    _shape("rowptr", rowptr, N + 1)
    _shape("x", x, N, t.d1, t.mul)
    _shape("y", y, E, t.d2)
    _radial_operands(t, E, h, W2)
    m = out if out is not None else torch.empty((N, t.D, t.mul), dtype=torch.float32, device=x.device)
    _shape("m", m, N, t.D, t.mul)
    _f32_out(m, h, W2)
    _check(load().e3gb_conv_forward_radial(t.handle, N, E, _ptr(rowptr), _ptr(sender) if E else None, _ptr(x),
                                           _ptr(y) if E else None, _ptr(h) if E else None, _ptr(W2), RADIAL_HIDDEN,
                                           float(scale), int(pad_node), _ptr(m), _dtype(x, *((y,) if E else ())),
                                           _stream(stream)))
    return m


def conv_backward_radial(t: Table, csc, x, y, h, W2, dm, scale: float, out=None, stream=None, pad_node: int = -1):
    """Returns (dx, dy, dh): conv_backward with dw folded into dh = sum_{p,q} W2 dw (dw never stored)."""
    import torch
    cp, ce, cr = csc
    _contig(x, y, h, W2, dm)
    N, E = x.shape[0], y.shape[0]
    _csc_shapes(csc, N, E)
    _shape("x", x, N, t.d1, t.mul)
    _shape("y", y, E, t.d2)
    _radial_operands(t, E, h, W2)
    _shape("dm", dm, N, t.D, t.mul)
    if out is None:
        f = dict(dtype=torch.float32)
        out = (torch.empty_like(x, **f), torch.empty_like(y, **f), torch.empty_like(h, **f))
    dx, dy, dh = out
    _shape("dx", dx, N, t.d1, t.mul)
    _shape("dy", dy, E, t.d2)
    _shape("dh", dh, E, RADIAL_HIDDEN)
    _f32_out(dx, dy, dh, h, W2)
    _check(load().e3gb_conv_backward_radial(t.handle, N, E, _ptr(cp), _ptr(ce) if E else None,
                                            _ptr(cr) if E else None, _ptr(x), _ptr(y) if E else None,
                                            _ptr(h) if E else None, _ptr(W2), RADIAL_HIDDEN, _ptr(dm), float(scale),
                                            int(pad_node), _ptr(dx), _ptr(dy) if E else None,
                                            _ptr(dh) if E else None, _dtype(x, dm, *((y,) if E else ())),
                                            _stream(stream)))
    return dx, dy, dh


def conv_double_backward(t: Table, rowptr, sender, csc, x, y, w, dm, delta_dx, delta_dy, delta_dw, scale: float,
                         out=None, stream=None, pad_node: int = -1):
    """Eq. (17)-(18): returns (delta_x, delta_y, delta_w, delta_dm), the gradient of
    <dx, delta_dx> + <dy, delta_dy> + <dw, delta_dw> over (x, y, w, dm)."""
    import torch
    cp, ce, cr = csc
    _contig(rowptr, sender, x, y, w, dm, delta_dx, delta_dy, delta_dw)
    N, E = x.shape[0], y.shape[0]
    _shape("rowptr", rowptr, N + 1)
    _shape("sender", sender, E)
    _csc_shapes(csc, N, E)
    _conv_operands(t, N, E, x, y, w)
    _conv_operands(t, N, E, delta_dx, delta_dy, delta_dw, ("delta_dx", "delta_dy", "delta_dw"))
    _shape("dm", dm, N, t.D, t.mul)
    if out is None:
        f = dict(dtype=torch.float32)
        out = (torch.empty_like(x, **f), torch.empty_like(y, **f), torch.empty_like(w, **f),
               torch.empty_like(dm, **f))
    gx, gy, gw, gdm = out
    _conv_operands(t, N, E, gx, gy, gw, ("delta_x", "delta_y", "delta_w"))
    _shape("delta_dm", gdm, N, t.D, t.mul)
    _f32_out(gx, gy, gw, gdm)
    e = (lambda a: _ptr(a) if E else None)
    _check(load().e3gb_conv_double_backward(
        t.handle, N, E, _ptr(rowptr), e(sender), _ptr(cp), e(ce), e(cr), _ptr(x), e(y), e(w), _ptr(dm),
        _ptr(delta_dx), e(delta_dy), e(delta_dw), float(scale), int(pad_node), _ptr(gx), e(gy), e(gw), _ptr(gdm),
        _dtype(x, dm, delta_dx, *((y, w, delta_dy, delta_dw) if E else ())), _stream(stream)))
    return gx, gy, gw, gdm


def coo_tp_forward(rec, coef, x, y, w, D: int, out=None, stream=None):
    """Tensor product with runtime COO coefficients: rec int32 [n,4] (i0, i1, i2, path) and
    coef fp32 [n] on the device; x [R,d1,mul], y [R,d2], w [R,P,mul] -> z [R,D,mul] fp32."""
    import torch
    _contig(rec, coef, x, y, w)
    R, d1, mul = x.shape
    z = out if out is not None else torch.empty((R, D, mul), dtype=torch.float32, device=x.device)
    _f32_out(z)
    n = rec.shape[0]
    _check(load().e3gb_coo_tp_forward(R, d1, y.shape[1], D, w.shape[1], mul, n, _ptr(rec) if n else None,
                                      _ptr(coef) if n else None, _ptr(x), _ptr(y), _ptr(w), _ptr(z), _dtype(x, y, w),
                                      _stream(stream)))
    return z


def coo_tp_backward(rec, coef, x, y, w, dz, out=None, stream=None):
    """(dx, dy, dw) of coo_tp_forward."""
    import torch
    _contig(rec, coef, x, y, w, dz)
    R, d1, mul = x.shape
    if out is None:
        f = dict(dtype=torch.float32)
        out = (torch.empty_like(x, **f), torch.empty_like(y, **f), torch.empty_like(w, **f))
    dx, dy, dw = out
    _f32_out(dx, dy, dw)
    n = rec.shape[0]
    _check(load().e3gb_coo_tp_backward(R, d1, y.shape[1], dz.shape[1], w.shape[1], mul, n, _ptr(rec) if n else None,
                                       _ptr(coef) if n else None, _ptr(x), _ptr(y), _ptr(w), _ptr(dz), _ptr(dx),
                                       _ptr(dy), _ptr(dw), _dtype(x, y, w, dz), _stream(stream)))
    return dx, dy, dw


def check_device_status(stream=None) -> int:
    """Synchronise and read/clear the device error word; raises E3GBError if it was set."""
    flags = ctypes.c_int32()
    st = load().e3gb_check_device_status(_stream(stream), ctypes.byref(flags))
    if st != OK:
        raise E3GBError(st, load().e3gb_last_error().decode())
    return flags.value


def shard_graphs(graph_ptr, rowptr, sender, world: int, rank: int) -> tuple[int, int, int, int]:
    """Data-parallel split of a batch of independent graphs (molecules) stored as one
    receiver-sorted CSR: graph g owns nodes [graph_ptr[g], graph_ptr[g+1]) and every edge into
    them, and each of its edges must come from one of its own nodes. Returns (n0, n1, e0, e1):
    rank's contiguous run of whole graphs, cut at the graph boundaries nearest to r * E / world
    so that the ranks' edge counts differ by at most about one graph's edges. The rank's own
    CSR is rowptr[n0:n1+1] - e0 with senders sender[e0:e1] - n0; no edge crosses ranks, so
    the ranks exchange nothing on the data path (host logic, numpy; raises ValueError if an
    edge leaves its graph)."""
    import numpy as np

    gp = np.asarray(graph_ptr, dtype=np.int64)
    rp = np.asarray(rowptr, dtype=np.int64)
    sd = np.asarray(sender, dtype=np.int64)
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    N, E = rp.shape[0] - 1, int(rp[-1]) if rp.shape[0] else 0
    if gp.ndim != 1 or gp.shape[0] < 1 or gp[0] != 0 or gp[-1] != N or np.any(np.diff(gp) < 0):
        raise ValueError("graph_ptr must rise from 0 to the node count")
    if rp[0] != 0 or np.any(np.diff(rp) < 0) or sd.shape[0] != E:
        raise ValueError("rowptr / sender do not form a CSR")
    # the graph of each edge's receiver and of its sender must agree
    recv = np.repeat(np.arange(N, dtype=np.int64), np.diff(rp))
    g_of = lambda v: np.searchsorted(gp, v, side="right") - 1
    if E and (np.any(sd < 0) or np.any(sd >= N) or np.any(g_of(recv) != g_of(sd))):
        raise ValueError("an edge joins two graphs: the batch cannot be split without a halo")
    eb = rp[gp]   # edge offset at each graph boundary (non-decreasing)
    cut = [0]
    for r in range(1, world):
        t = r * E / world
        b = int(np.searchsorted(eb, t))
        if b > 0 and (b >= eb.shape[0] or t - eb[b - 1] <= eb[b] - t):
            b -= 1
        cut.append(max(b, cut[-1]))
    cut.append(gp.shape[0] - 1)
    n0, n1 = int(gp[cut[rank]]), int(gp[cut[rank + 1]])
    return n0, n1, int(rp[n0]), int(rp[n1])
