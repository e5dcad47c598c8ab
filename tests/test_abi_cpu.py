"""The C-ABI library without a GPU: it loads, exports every symbol include/e3gb.h declares,
and its host-side path tables and CG records agree with the oracle's (an independent
construction: ladder operators of App. G.2 in the library, a null-space solve in the
oracle)."""
import ctypes
import os
import re

import numpy as np
import pytest

import message_passing_gb300 as e3
import oracle
from oracle.cg import cg_block

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONFIGS = [
    ([(0, 1), (1, -1)], 16, 2, 2, False),
    ([(0, 1), (1, -1), (2, 1)], 128, 3, 3, False),
    ([(0, 1), (1, -1)], 128, 3, 3, False),
    ([(0, 1), (1, -1), (2, 1), (3, -1)], 8, 3, 3, False),
    ([(0, 1)], 4, 0, 0, False),
    ([(1, -1)], 4, 1, 2, True),
    ([(0, 1), (1, -1)], 16, 2, 2, True),
    ([(0, 1), (1, -1), (2, 1)], 128, 3, 3, True),
]


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(e3.LIB_PATH):
        from message_passing_gb300 import build
        build.build()
    return e3.load()


def test_exports_every_declared_symbol(lib):
    hdr = open(os.path.join(ROOT, "include", "e3gb.h")).read()
    declared = set(re.findall(r"\b(e3gb_[a-z_0-9]+)\s*\(", hdr))
    assert declared == set(e3.SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_configs(lib):
    assert "sm_103a" in e3.version()
    cfgs = e3.configs()
    assert len(cfgs) == len(CONFIGS)
    for blocks, _, L2, L3, pp in CONFIGS:
        assert {"blocks": blocks, "sh_lmax": L2, "out_lmax": L3, "per_path": pp} in cfgs


@pytest.mark.parametrize("blocks,mul,L2,L3,pp", CONFIGS)
def test_table_matches_oracle(lib, blocks, mul, L2, L3, pp):
    t = e3.Table.create(blocks, mul, L2, L3, pp)
    ot = oracle.table(blocks, L2, L3, pp)
    assert (t.d1, t.d2, t.n_paths, t.D) == (ot.d1, ot.d2, ot.n_paths, ot.D)
    got = t.paths()
    want = [(p.xblock, p.l1, p.p1, p.l2, p.l3, p.p3, p.out_block, p.zoff) for p in ot.paths]
    assert got == want
    rec = t.coefficients()
    assert rec.shape[0] == sum(int((cg_block(p.l1, p.l2, p.l3) != 0).sum()) for p in ot.paths)
    for path, m1, m2, m3, v in rec:
        p = ot.paths[int(path)]
        assert abs(cg_block(p.l1, p.l2, p.l3)[int(m1), int(m2), int(m3)] - v) < 1e-12


def test_table_errors(lib):
    with pytest.raises(e3.E3GBError) as ex:
        e3.Table.create([(2, 1)], 16, 3, 3)
    assert ex.value.status == e3.ERR_UNSUPPORTED
    with pytest.raises(e3.E3GBError) as ex:
        e3.Table.create([(0, 1), (1, -1)], 12, 2, 2)
    assert ex.value.status == e3.ERR_UNSUPPORTED
    with pytest.raises(e3.E3GBError) as ex:
        e3.Table.create([(0, 0)], 16, 0, 0)
    assert ex.value.status == e3.ERR_INVALID_ARG
    with pytest.raises(e3.E3GBError) as ex:
        e3.Table.create([(0, 1)], 16, 4, 0)
    assert ex.value.status == e3.ERR_UNSUPPORTED


def test_host_argument_checks_need_no_gpu(lib):
    """Null pointers and bad sizes are rejected before any CUDA call."""
    t = e3.Table.create([(0, 1), (1, -1)], 16, 2, 2)
    assert lib.e3gb_tp_forward(t.handle.value, 0, None, None, None, None, 0, None) == e3.OK
    assert lib.e3gb_tp_forward(t.handle.value, 4, None, None, None, None, 0, None) == e3.ERR_INVALID_ARG
    assert b"NULL" in lib.e3gb_last_error()
    assert lib.e3gb_tp_forward(t.handle.value, -1, None, None, None, None, 0, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_tp_forward(t.handle.value, 4, None, None, None, None, 7, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_conv_forward(t.handle.value, 0, 5, None, None, None, None, None, ctypes.c_float(1.0), -1,
                                 None, 0, None) == e3.ERR_BAD_GRAPH
    # the padding node must be a node (or -1 for none)
    for pad in (-2, 4, 100):
        assert lib.e3gb_conv_forward(t.handle.value, 4, 5, None, None, None, None, None, ctypes.c_float(1.0), pad,
                                     None, 0, None) == e3.ERR_INVALID_ARG
        assert b"pad_node" in lib.e3gb_last_error()
        assert lib.e3gb_conv_backward(t.handle.value, 4, 5, None, None, None, None, None, None, None,
                                      ctypes.c_float(1.0), pad, None, None, None, 0, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_sh_forward(4, 3, None, None, 0, None) == e3.ERR_UNSUPPORTED
    assert lib.e3gb_graph_prepare(10, 20, None, None, None, None, None, None, 0, None) == e3.ERR_INVALID_ARG
    # one 256-entry digit count per tile of 1024 edges, plus the scan's block sums
    assert lib.e3gb_graph_prepare_workspace_bytes(1000, 5000) >= 256 * 5 * 4
    assert lib.e3gb_graph_prepare_workspace_bytes(1000, 0) >= 0


def test_radial_argument_checks_need_no_gpu(lib):
    """The radial entry points reject bad network sizes, other dtypes and other hidden widths
    on the host."""
    f = ctypes.c_float
    assert lib.e3gb_radial_hidden(0, None, None, 0, 8, f(4.0), None, None) == e3.ERR_INVALID_ARG
    assert b"n_basis" in lib.e3gb_last_error()
    assert lib.e3gb_radial_hidden(0, None, None, 8, 17, f(4.0), None, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_radial_hidden(0, None, None, 8, 8, f(0.0), None, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_radial_backward(5, None, None, 8, 8, f(4.0), None, None, 0, None) == e3.ERR_INVALID_ARG
    t = e3.Table.create([(0, 1), (1, -1)], 16, 2, 2)
    # bf16 and hidden widths other than the compiled one are not built
    assert lib.e3gb_conv_forward_radial(t.handle.value, 4, 5, None, None, None, None, None, None, 8, f(1.0), -1,
                                        None, e3.BF16, None) == e3.ERR_UNSUPPORTED
    assert lib.e3gb_conv_forward_radial(t.handle.value, 4, 5, None, None, None, None, None, None, 4, f(1.0), -1,
                                        None, e3.F32, None) == e3.ERR_UNSUPPORTED
    assert lib.e3gb_conv_backward_radial(t.handle.value, 4, 5, None, None, None, None, None, None, None, 16, None,
                                         f(1.0), -1, None, None, None, e3.F32, None) == e3.ERR_UNSUPPORTED
    assert lib.e3gb_conv_forward_radial(t.handle.value, 4, 5, None, None, None, None, None, None, 8, f(1.0), 9,
                                        None, e3.F32, None) == e3.ERR_INVALID_ARG
    assert lib.e3gb_conv_forward_radial(t.handle.value, 4, 5, None, None, None, None, None, None, 8, f(1.0), -1,
                                        None, e3.F32, None) == e3.ERR_INVALID_ARG
    assert b"NULL" in lib.e3gb_last_error()


def test_split_forward_argument_checks_need_no_gpu(lib):
    f = ctypes.c_float
    t = e3.Table.create([(0, 1), (1, -1)], 16, 2, 2)
    # workspace: piece pointers and scan sums for N + 1 entries, E / chunk + 1 partial row sets
    nb = lib.e3gb_conv_forward_split_workspace_bytes(t.handle.value, 100, 5000, 64)
    assert nb >= (5000 // 64 + 1) * t.D * t.mul * 4
    assert lib.e3gb_conv_forward_split_workspace_bytes(t.handle.value, 100, 5000, 0) == 0
    args = lambda chunk, ws: (t.handle.value, 4, 5, None, None, None, None, None, f(1.0), -1, chunk, None, None, ws,
                              e3.F32, None)
    assert lib.e3gb_conv_forward_split(*args(0, 1 << 20)) == e3.ERR_INVALID_ARG
    assert b"chunk" in lib.e3gb_last_error()
    assert lib.e3gb_conv_forward_split(*args(8, 16)) == e3.ERR_INVALID_ARG
    assert b"workspace" in lib.e3gb_last_error()
    # one output block per path on 0e+1o+2e: 106 rows per receiver, not built for the split form
    tp = e3.Table.create([(0, 1), (1, -1), (2, 1)], 128, 3, 3, per_path=True)
    assert tp.D == 106
    assert lib.e3gb_conv_forward_split(tp.handle.value, 4, 5, None, None, None, None, None, f(1.0), -1, 8, None, None,
                                       1 << 30, e3.F32, None) == e3.ERR_UNSUPPORTED


def test_table_coo_records_match_the_oracle_records():
    """The binding's CG records (library table, host side) are the oracle's CG records up to
    order and rounding to fp32."""
    import numpy as np
    import oracle
    blocks = [(0, 1), (1, -1), (2, 1)]
    t = e3.Table.create(blocks, 128, 3, 3)
    rec, c = t.coo_records()
    orec, oc = oracle.cg_records(oracle.table(blocks, 3, 3))
    key = lambda r: np.lexsort(r.T[::-1])
    a, b = key(rec), key(orec)
    assert np.array_equal(rec[a], orec[b])
    np.testing.assert_allclose(c[a], oc[b], rtol=1e-6, atol=1e-7)
