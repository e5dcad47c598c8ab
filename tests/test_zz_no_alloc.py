"""The allocation-free graph index entry point, e3gb_graph_prepare_static.

It serves callers that must not allocate device memory (a host that gave all free memory
to its own pool, a plugin whose host owns every allocation, a latency-critical loop that
cannot take cudaMalloc's device-wide synchronisation): the sort's digit counts live in a
static array inside the library instead of a caller workspace. Its result must equal that
of e3gb_graph_prepare bit for bit, on consecutive calls (the array keeps the previous
call's contents, which no call may depend on). This file sorts last so that a run
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


def test_static_prepare_large_graph_with_longer_tiles(cuda):
    """More than a million nodes and ~4.5 M edges: the library's array holds the counts of
    ~4,000 tiles, so each tile covers 2,048 edges here (1,024 with a workspace). One edge
    leaves the last node and one enters it. The result must still equal the workspace
    entry point's bit for bit, and numpy's stable argsort."""
    e3.load()
    N, E = 1_200_000, 4_500_000
    rng = np.random.default_rng(97)
    recv = np.sort(rng.integers(0, N, E))
    send = rng.integers(0, N, E)
    send[E // 2] = N - 1
    recv[-1] = N - 1
    rowptr = np.zeros(N + 1, np.int64)
    np.cumsum(np.bincount(recv, minlength=N), out=rowptr[1:])
    rp = torch.from_numpy(rowptr.astype(np.int32)).cuda()
    sd = torch.from_numpy(send.astype(np.int32)).cuda()
    want = e3.graph_prepare(rp, sd, N)
    for _ in range(2):
        got = _static(rp, sd, N)
        torch.cuda.synchronize()
        assert e3.check_device_status() == 0
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    order = np.argsort(send, kind="stable")
    assert np.array_equal(got[1].cpu().numpy(), order)
    assert np.array_equal(got[2].cpu().numpy(), recv[order])
    assert int(got[0][N - 1]) == E - int((send == N - 1).sum())


def test_static_prepare_rejects_oversized_graphs(cuda):
    lib = e3.load()
    st = lib.e3gb_graph_prepare_static(2 ** 31 - 1, 0, None, None, None, None, None, None)
    assert st == e3.ERR_INVALID_ARG
    assert b"e3gb_graph_prepare_static" in lib.e3gb_last_error()
