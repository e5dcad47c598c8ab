"""Pins of the oracle's padding-edge rule (oracle.conv_forward / conv_backward_* with pad_node).

e3j, Sec. 4 "Message passing convolution" and App. E: static-shape graphs send their unused
edge slots to one padding node and the convolution kernels skip those edges. The pin is the
unpadded graph itself: adding a padding node and padding edges (pad -> pad, pad -> real,
real -> pad) with NaN inputs, and naming pad_node, must leave every real output bit for bit
what the plain conv of the original graph gives, with zeros for the padding rows.
"""
import numpy as np
import pytest

import oracle
import synth

IRREPS = [(0, 1), (1, -1)]


@pytest.mark.parametrize("n_self,n_out,n_in", [(40, 0, 0), (25, 9, 7), (0, 0, 5)])
def test_padding_equals_unpadded_graph(n_self, n_out, n_in):
    t = oracle.table(IRREPS, 2, 2)
    g = synth.random_graph(30, 160, (77, 0), empty_nodes=3)
    gp, pad, orig = synth.padded_graph(g, n_self, n_out, n_in, (77, 1))
    assert gp.n_edges == g.n_edges + n_self + n_out + n_in and pad == g.n_nodes
    r = np.random.default_rng(5)
    Nq, E = 4, g.n_edges
    x = r.standard_normal((g.n_nodes, t.d1, Nq))
    y = r.standard_normal((E, t.d2))
    w = r.standard_normal((E, t.n_paths, Nq))
    dm = r.standard_normal((g.n_nodes, t.D, Nq))
    real = orig >= 0
    # padded inputs: real rows copied, every padding row and the padding node's rows NaN
    xp = np.concatenate([x, np.full((1, t.d1, Nq), np.nan)])
    dmp = np.concatenate([dm, np.full((1, t.D, Nq), np.nan)])
    yp = np.full((gp.n_edges, t.d2), np.nan); yp[real] = y[orig[real]]
    wp = np.full((gp.n_edges, t.n_paths, Nq), np.nan); wp[real] = w[orig[real]]

    m = oracle.conv_forward(t, g.rowptr, g.sender, x, y, w, 0.5)
    mp = oracle.conv_forward(t, gp.rowptr, gp.sender, xp, yp, wp, 0.5, pad_node=pad)
    np.testing.assert_array_equal(mp[:-1], m)
    assert np.all(mp[pad] == 0.0)

    dy, dw = oracle.conv_backward_edges(t, g.rowptr, g.sender, x, y, w, dm, 0.5)
    dyp, dwp = oracle.conv_backward_edges(t, gp.rowptr, gp.sender, xp, yp, wp, dmp, 0.5, pad_node=pad)
    np.testing.assert_array_equal(dyp[real], dy[orig[real]])
    np.testing.assert_array_equal(dwp[real], dw[orig[real]])
    assert np.all(dyp[~real] == 0.0) and np.all(dwp[~real] == 0.0)

    dx = oracle.conv_backward_dx(t, g.rowptr, g.sender, y, w, dm, 0.5, Nq=Nq)
    dxp = oracle.conv_backward_dx(t, gp.rowptr, gp.sender, yp, wp, dmp, 0.5, Nq=Nq, pad_node=pad)
    np.testing.assert_array_equal(dxp[:-1], dx)
    assert np.all(dxp[pad] == 0.0)


def test_padding_rule_is_not_vacuous():
    """Without pad_node the NaN padding rows reach the outputs (the rule does the skipping)."""
    t = oracle.table(IRREPS, 2, 2)
    g = synth.random_graph(12, 40, (78, 0))
    gp, pad, orig = synth.padded_graph(g, 5, 3, 3, (78, 1))
    xp = np.concatenate([np.ones((12, t.d1, 2)), np.full((1, t.d1, 2), np.nan)])
    yp = np.ones((gp.n_edges, t.d2)); wp = np.ones((gp.n_edges, t.n_paths, 2))
    m = oracle.conv_forward(t, gp.rowptr, gp.sender, xp, yp, wp, 1.0)
    assert np.isnan(m).any()
    assert not np.isnan(oracle.conv_forward(t, gp.rowptr, gp.sender, xp, yp, wp, 1.0, pad_node=pad)).any()
