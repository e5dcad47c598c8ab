"""The Python binding refuses buffers whose shapes do not match the path table and the
row/node/edge counts, on the host and before any library call: the kernels index every
buffer from those sizes, so a smaller buffer would be read or written out of bounds."""
import os

import pytest
import torch

import message_passing_gb300 as e3


@pytest.fixture(scope="module")
def table():
    if not os.path.exists(e3.LIB_PATH):
        from message_passing_gb300 import build
        build.build()
    e3.load()
    return e3.Table.create([(0, 1), (1, -1), (2, 1)], 8, 3, 3)   # d1 9, d2 16, 24 paths, D 31


N, E = 5, 7


def _conv(t):
    return dict(rowptr=torch.zeros(N + 1, dtype=torch.int32), sender=torch.zeros(E, dtype=torch.int32),
                x=torch.zeros(N, t.d1, t.mul), y=torch.zeros(E, t.d2), w=torch.zeros(E, t.n_paths, t.mul))


def test_table_sizes(table):
    assert (table.d1, table.d2, table.n_paths, table.D, table.mul) == (9, 16, 24, 31, 8)


@pytest.mark.parametrize("name,shape", [("x", (N, 8, 8)), ("x", (N, 9, 4)), ("y", (E - 1, 16)), ("y", (E, 9)),
                                        ("w", (E, 23, 8)), ("w", (E + 1, 24, 8)), ("rowptr", (N,))])
def test_conv_forward_rejects(table, name, shape):
    a = _conv(table)
    a[name] = torch.zeros(shape, dtype=a[name].dtype)
    with pytest.raises(ValueError, match=name):
        e3.conv_forward(table, a["rowptr"], a["sender"], a["x"], a["y"], a["w"], 1.0)


def test_conv_forward_rejects_output(table):
    a = _conv(table)
    with pytest.raises(ValueError, match="m"):
        e3.conv_forward(table, a["rowptr"], a["sender"], a["x"], a["y"], a["w"], 1.0,
                        out=torch.zeros(N, table.D - 1, table.mul))


def test_conv_backward_rejects(table):
    a = _conv(table)
    csc = (torch.zeros(N + 1, dtype=torch.int32), torch.zeros(E, dtype=torch.int32), torch.zeros(E, dtype=torch.int32))
    dm = torch.zeros(N, table.D, table.mul)
    with pytest.raises(ValueError, match="dm"):
        e3.conv_backward(table, csc, a["x"], a["y"], a["w"], torch.zeros(N, table.D, 4), 1.0)
    with pytest.raises(ValueError, match="csc_edge"):
        short = (csc[0], torch.zeros(E - 1, dtype=torch.int32), csc[2])
        e3.conv_backward(table, short, a["x"], a["y"], a["w"], dm, 1.0)
    with pytest.raises(ValueError, match="csc_ptr"):
        e3.conv_backward(table, (torch.zeros(N, dtype=torch.int32), csc[1], csc[2]), a["x"], a["y"], a["w"], dm, 1.0)
    with pytest.raises(ValueError, match="dw"):
        out = (torch.zeros_like(a["x"]), torch.zeros_like(a["y"]), torch.zeros(E, 2, table.mul))
        e3.conv_backward(table, csc, a["x"], a["y"], a["w"], dm, 1.0, out=out)


def test_conv_double_backward_rejects(table):
    a = _conv(table)
    csc = (torch.zeros(N + 1, dtype=torch.int32), torch.zeros(E, dtype=torch.int32), torch.zeros(E, dtype=torch.int32))
    dm = torch.zeros(N, table.D, table.mul)
    with pytest.raises(ValueError, match="delta_dw"):
        e3.conv_double_backward(table, a["rowptr"], a["sender"], csc, a["x"], a["y"], a["w"], dm,
                                torch.zeros_like(a["x"]), torch.zeros_like(a["y"]), torch.zeros(E, 3, table.mul), 1.0)


def test_tp_rejects(table):
    R = 6
    x, y, w = torch.zeros(R, table.d1, table.mul), torch.zeros(R, table.d2), torch.zeros(R, table.n_paths, table.mul)
    with pytest.raises(ValueError, match="w"):
        e3.tp_forward(table, x, y, torch.zeros(R - 1, table.n_paths, table.mul))
    with pytest.raises(ValueError, match="z"):
        e3.tp_forward(table, x, y, w, out=torch.zeros(R, table.D, 4))
    with pytest.raises(ValueError, match="dz"):
        e3.tp_backward(table, x, y, w, torch.zeros(R, table.D - 1, table.mul))


def test_sh_and_graph_prepare_reject():
    with pytest.raises(ValueError, match="vec"):
        e3.sh_forward(torch.zeros(4, 4), 3)
    with pytest.raises(ValueError, match="dy"):
        e3.sh_backward(torch.zeros(4, 3), torch.zeros(4, 9), 3)
    with pytest.raises(ValueError, match="rowptr"):
        e3.graph_prepare(torch.zeros(N, dtype=torch.int32), torch.zeros(E, dtype=torch.int32), N)
    with pytest.raises(ValueError, match="csc_recv"):
        out = (torch.zeros(N + 1, dtype=torch.int32), torch.zeros(E, dtype=torch.int32),
               torch.zeros(E - 2, dtype=torch.int32))
        e3.graph_prepare_static(torch.zeros(N + 1, dtype=torch.int32), torch.zeros(E, dtype=torch.int32), N, out=out)
