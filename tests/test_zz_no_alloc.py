"""The allocation-free graph index entry point, e3gb_graph_prepare_static.

It serves callers that must not allocate device memory (a host that gave all free memory
to its own pool, a plugin whose host owns every allocation, a latency-critical loop that
cannot take cudaMalloc's device-wide synchronisation): the per-node counters live in a
static array inside the library instead of a caller workspace. Its result must equal that
of e3gb_graph_prepare bit for bit, on consecutive calls (the array keeps the previous
call's contents and has to be cleared by each call). This file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
from synth import random_graph
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _static(rp, sd, n_nodes):
    """Call the entry point through the C ABI, with caller-owned outputs."""
    lib = e3.load()
    E = sd.numel()
    cp = torch.full((n_nodes + 1,), -7, dtype=torch.int32, device="cuda")
    ce = torch.full((max(E, 1),), -7, dtype=torch.int32, device="cuda")
    cr = torch.full((max(E, 1),), -7, dtype=torch.int32, device="cuda")
    st = lib.e3gb_graph_prepare_static(n_nodes, E, ctypes.c_void_p(rp.data_ptr()),
                                       ctypes.c_void_p(sd.data_ptr() if E else 0),
                                       ctypes.c_void_p(cp.data_ptr()), ctypes.c_void_p(ce.data_ptr()),
                                       ctypes.c_void_p(cr.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == e3.OK, lib.e3gb_last_error()
    return cp, ce, cr


def test_static_prepare_equals_workspace_prepare(cuda):
    e3.load()
    big = W.make_graph(W.WORKLOADS[3])                                   # 4096 atoms, ~214k edges
    small = random_graph(700, 9000, (96, 1), empty_nodes=50)             # smaller, after the big one
    for g in (big, small):
        rp = torch.from_numpy(g.rowptr).cuda()
        sd = torch.from_numpy(g.sender).cuda()
        want = e3.graph_prepare(rp, sd, g.n_nodes)
        got = _static(rp, sd, g.n_nodes)
        torch.cuda.synchronize()
        assert e3.check_device_status() == 0
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        order = np.argsort(g.sender, kind="stable")
        assert np.array_equal(got[1].cpu().numpy(), order)


def test_static_prepare_rejects_too_many_nodes(cuda):
    lib = e3.load()
    st = lib.e3gb_graph_prepare_static(e3.STATIC_PREPARE_MAX_NODES + 1, 0, None, None, None, None, None, None)
    assert st == e3.ERR_INVALID_ARG
    assert b"static scratch" in lib.e3gb_last_error()
