"""bench.py's byte accounting and traffic bookkeeping, on the CPU.

The algorithmic bytes follow "e3j ...", Sec. 3 Eq. (9): the bytes of every input and output
array of a call (the backward counts input primals, output cotangents and input cotangents).
Here they are checked against the sizes of actual arrays of those shapes, and the per-kernel
source hash that keys profiles/traffic.json against edits of the files it covers.
"""
import numpy as np

import bench


def _nbytes(*arrays):
    return sum(a.nbytes for a in arrays)


def test_conv_bytes_are_the_arrays_of_a_call():
    N, E, d1, d2, P, D, Nq = 37, 211, 9, 16, 24, 31, 8
    for dt, s in ((np.float32, 4), (np.float16, 2)):   # float16 stands in for any 2-byte storage
        x, y, w, dm = (np.zeros(sh, dt) for sh in ((N, d1, Nq), (E, d2), (E, P, Nq), (N, D, Nq)))
        rowptr, sender = np.zeros(N + 1, np.int32), np.zeros(E, np.int32)
        csc_ptr, csc_edge, csc_recv = np.zeros(N + 1, np.int32), np.zeros(E, np.int32), np.zeros(E, np.int32)
        m = np.zeros((N, D, Nq), np.float32)
        dx, dy, dw = (np.zeros(sh, np.float32) for sh in ((N, d1, Nq), (E, d2), (E, P, Nq)))
        fwd, bwd = bench.conv_bytes(N, E, d1, d2, P, D, Nq, s)
        assert fwd == _nbytes(x, y, w, rowptr, sender, m)
        assert bwd == _nbytes(x, y, w, dm, csc_ptr, csc_edge, csc_recv, dx, dy, dw)


def test_conv_bytes_per_edge_of_the_64k_workload():
    """12.87 KB (forward) and 25.34 KB (backward) per edge, the figures the roofline uses."""
    N, E = 64000, 2558876
    fwd, bwd = bench.conv_bytes(N, E, 9, 16, 24, 31, 128, 4)
    assert abs(fwd / E - 12868) < 1
    assert abs(bwd / E - 25340) < 1


def test_tp_bytes_are_the_arrays_of_a_call():
    R, d1, d2, P, D, Nq = 53, 4, 9, 9, 17, 16
    x, y, w, z = (np.zeros(sh, np.float32) for sh in ((R, d1, Nq), (R, d2), (R, P, Nq), (R, D, Nq)))
    dx, dy, dw = np.zeros_like(x), np.zeros_like(y), np.zeros_like(w)
    fwd, bwd = bench.tp_bytes(R, d1, d2, P, D, Nq, 4)
    assert fwd == _nbytes(x, y, w, z)
    assert bwd == _nbytes(x, y, w, z, dx, dy, dw)   # dz has the shape of z


def test_sh_bytes():
    E = 101
    assert bench.sh_bytes(E, 16, 4) == _nbytes(np.zeros((E, 3), np.float32), np.zeros((E, 16), np.float32))


def test_kernel_source_hash_covers_only_the_kernels_files(tmp_path, monkeypatch):
    csrc = tmp_path / "message_passing_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for n in ("conv_pipe.cuh", "kernels.cuh", "cg_table.hpp", "configs.def", "instances.cu", "sh.cu"):
        (csrc / n).write_text(n)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0, a0 = bench.kernel_source_hash("conv_bwd"), bench.kernel_source_hash()
    (csrc / "sh.cu").write_text("changed")                 # not a source of the conv kernels
    assert bench.kernel_source_hash("conv_bwd") == h0
    assert bench.kernel_source_hash() != a0
    (csrc / "conv_pipe.cuh").write_text("changed")         # one of them
    assert bench.kernel_source_hash("conv_bwd") != h0
