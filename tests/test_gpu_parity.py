"""Parity of every CUDA entry point with the float64 oracle.

Tolerances (per output tensor): max |err| <= 1e-5 RMS(oracle) for fp32 I/O and 2e-2 RMS for
bf16 storage. Inputs are the seeded workloads of synth.workloads: small cases compared
element by element, full-size cases on sampled rows / receivers / senders / edges computed
one by one by the oracle.
"""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
from gpu_util import TOL_BF16, TOL_F32, assert_close, sample_ids, to_dev, to_np
from synth import STREAM_GRAD, STREAM_W, device_normal, random_graph
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _tables(w, per_path=False):
    return (e3.Table.create(w.blocks, w.mul, w.sh_lmax, w.out_lmax, per_path),
            oracle.table(w.blocks, w.sh_lmax, w.out_lmax, per_path))


# ------------------------------------------------------------------------------------------
# spherical harmonics
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("lmax", [0, 1, 2, 3])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_sh(lmax, dt):
    rng = np.random.default_rng(lmax)
    vec = rng.standard_normal((1037, 3)) * rng.uniform(0.1, 6.0, (1037, 1))
    vec[0] = 0.0                       # zero vector: Y_0 = 1, others 0
    vec[1] = (0.0, 0.0, 3.0)
    vec[2] = (-2.0, 0.0, 0.0)
    v32 = vec.astype(np.float32)
    y = e3.sh_forward(to_dev(v32), lmax, dtype=dt)
    torch.cuda.synchronize()
    ref = oracle.sh(v32.astype(np.float64), lmax)
    assert_close(to_np(y), ref, TOL_F32 if dt == torch.float32 else TOL_BF16, f"Y l<={lmax}")
    assert to_np(y)[0, 0] == 1.0 and np.all(to_np(y)[0, 1:] == 0.0)


# ------------------------------------------------------------------------------------------
# tensor product on rows
# ------------------------------------------------------------------------------------------
def _tp_check(w, rows, per_path=False, row_ids=None, k_sample=None):
    t, ot = _tables(w, per_path)
    u, x, ww = W.make_tp(w, ot.n_paths, rows=rows)
    v32 = u.astype(np.float32)
    dz = W.make_grad(w, x.shape[0], ot.D)
    xd, wd, dzd = to_dev(x), to_dev(ww), to_dev(dz)
    y = e3.sh_forward(to_dev(v32), w.sh_lmax)
    z = e3.tp_forward(t, xd, y, wd)
    dx, dy, dw = e3.tp_backward(t, xd, y, wd, dzd)
    torch.cuda.synchronize()
    ids = np.arange(x.shape[0]) if k_sample is None else sample_ids(x.shape[0], k_sample, 7)
    ysh = oracle.sh(v32[ids].astype(np.float64), w.sh_lmax)
    ref = oracle.tp_forward(ot, x[ids], ysh, ww[ids])
    assert_close(to_np(z[torch.from_numpy(ids).cuda()]), ref, TOL_F32, "z")
    rdx, rdy, rdw = oracle.tp_backward(ot, x[ids], ysh, ww[ids], dz[ids])
    sel = torch.from_numpy(ids).cuda()
    assert_close(to_np(dx[sel]), rdx, TOL_F32, "dx")
    assert_close(to_np(dy[sel]), rdy, TOL_F32, "dy")
    assert_close(to_np(dw[sel]), rdw, TOL_F32, "dw")


def test_tp_small_workload():
    """1024 rows, 16x0e+16x1o, SH l<=2, outputs l<=2, w ~ N(0,1)."""
    _tp_check(W.WORKLOADS[1], None)


def test_tp_batched_reduced_rows():
    """128x0e+128x1o+128x2e, SH l<=3: 2093 rows (many blocks, ragged tail)."""
    _tp_check(W.WORKLOADS[2], 2093)


def test_tp_batched_full_size_sampled():
    """All 200,000 rows computed on the GPU; 256 rows checked against the oracle."""
    _tp_check(W.WORKLOADS[2], None, k_sample=256)


def test_tp_per_path_outputs():
    w = W.Workload(91, "per-path", "tp", "16x0e+16x1o", 2, 2, rows=333)
    _tp_check(w, None, per_path=True)


def test_tp_closed_form_config():
    w = W.Workload(92, "l1 only", "tp", "4x1o", 1, 2, rows=101)
    _tp_check(w, None, per_path=True)


@pytest.mark.parametrize("mul", [4, 8, 16, 32, 64, 128])
def test_tp_channel_counts(mul):
    w = W.Workload(93, "channels", "tp", f"{mul}x0e+{mul}x1o", 3, 3, rows=157)
    _tp_check(w, None)


# ------------------------------------------------------------------------------------------
# convolution
# ------------------------------------------------------------------------------------------
def _conv_gpu(t, rowptr, sender, vec32, x, ww, dm, scale, dtype=torch.float32, y=None):
    rp, sd = to_dev(rowptr), to_dev(sender)
    if y is None:
        y = e3.sh_forward(to_dev(vec32), t.sh_lmax, dtype=dtype)
    xd = x if torch.is_tensor(x) else to_dev(x, dtype)
    wd = ww if torch.is_tensor(ww) else to_dev(ww, dtype)
    dmd = dm if torch.is_tensor(dm) else to_dev(dm, dtype)
    m = e3.conv_forward(t, rp, sd, xd, y, wd, scale)
    csc = e3.graph_prepare(rp, sd, len(rowptr) - 1)
    dx, dy, dw = e3.conv_backward(t, csc, xd, y, wd, dmd, scale)
    assert e3.check_device_status() == 0
    return m, dx, dy, dw


def _conv_check(w, g, tol=TOL_F32, k_nodes=None, k_edges=None, dtype=torch.float32, device_w=False,
                per_path=False):
    t, ot = _tables(w, per_path)
    N, E = g.n_nodes, g.n_edges
    scale = N / max(E, 1)
    x, _ = W.make_conv(w, g, ot.n_paths, edge_ids=np.zeros(0, np.int64))
    if device_w:
        wd = device_normal((E, ot.n_paths, w.mul), (w.wid, STREAM_W), W.weight_scale(w, ot.n_paths), dtype=dtype)
        dmd = device_normal((N, ot.D, w.mul), (w.wid, STREAM_GRAD), dtype=dtype)
    else:
        _, wn = W.make_conv(w, g, ot.n_paths)
        wd, dmd = to_dev(wn, dtype), to_dev(W.make_grad(w, N, ot.D), dtype)
    xd = to_dev(x, dtype)
    vec32 = g.vec.astype(np.float32)
    yo = oracle.sh(vec32.astype(np.float64), w.sh_lmax)
    yd = None
    if dtype == torch.bfloat16:
        # both sides take the same stored bf16 harmonics: rounding the GPU's and the oracle's
        # harmonics to bf16 separately can differ by one bf16 step where a value sits at a
        # rounding midpoint (the SH kernel is checked on its own)
        yb = torch.from_numpy(yo.astype(np.float32)).to(torch.bfloat16)
        yo = to_np(yb)
        yd = yb.cuda()
    m, dx, dy, dw = _conv_gpu(t, g.rowptr, g.sender, vec32, xd, wd, dmd, scale, dtype, y=yd)
    torch.cuda.synchronize()
    # the oracle reads exactly the stored (possibly bf16-rounded) inputs, widened to f64
    xo = to_np(xd)
    dmo = to_np(dmd)
    wfetch = lambda ids: to_np(wd[torch.from_numpy(np.asarray(ids, np.int64)).cuda()])
    nodes = np.arange(N) if k_nodes is None else sample_ids(N, k_nodes, 11)
    edges = np.arange(E) if k_edges is None else sample_ids(E, k_edges, 12)
    sel_n = torch.from_numpy(nodes).cuda()
    sel_e = torch.from_numpy(edges).cuda()
    ref_m = oracle.conv_forward(ot, g.rowptr, g.sender, xo, yo, wfetch, scale, receivers=nodes)
    assert_close(to_np(m[sel_n]), ref_m, tol, "m")
    ref_dx = oracle.conv_backward_dx(ot, g.rowptr, g.sender, yo, wfetch, dmo, scale, senders=nodes, Nq=w.mul)
    assert_close(to_np(dx[sel_n]), ref_dx, tol, "dx")
    ref_dy, ref_dw = oracle.conv_backward_edges(ot, g.rowptr, g.sender, xo, yo, wfetch, dmo, scale, edges=edges)
    assert_close(to_np(dy[sel_e]), ref_dy, tol, "dy")
    assert_close(to_np(dw[sel_e]), ref_dw, tol, "dw")


def test_conv_reduced_box():
    """128x0e+128x1o, SH l<=3, rc = 5 A at 0.1 atoms/A^3 (the 4096-atom workload's geometry),
    400 atoms: every output compared."""
    w = W.WORKLOADS[3]
    _conv_check(w, W.make_graph(w, n_atoms=400))


def test_conv_full_size_sampled():
    """4096 atoms, ~214k edges, every receiver computed; 192 nodes and 512 edges checked."""
    w = W.WORKLOADS[3]
    _conv_check(w, W.make_graph(w), k_nodes=192, k_edges=512)


def test_conv_random_atom_order():
    w = W.WORKLOADS[3]
    _conv_check(w, W.make_graph(w, n_atoms=300, order="draw"))


def test_conv_mace_like_reduced():
    """128x0e+128x1o+128x2e, ~40 neighbours, 500 atoms: every output compared."""
    w = W.WORKLOADS[4]
    _conv_check(w, W.make_graph(w, n_atoms=500))


def test_conv_mace_like_full_size_fp32():
    """64,000 atoms, ~2.56M edges (the benchmark launch), sampled outputs."""
    w = W.WORKLOADS[4]
    _conv_check(w, W.make_graph(w), k_nodes=96, k_edges=384, device_w=True)
    torch.cuda.empty_cache()


def test_conv_mace_like_full_size_bf16():
    """Same, bf16 storage / fp32 accumulation; oracle reads the bf16-rounded inputs."""
    w = W.WORKLOADS[4]
    _conv_check(w, W.make_graph(w), tol=TOL_BF16, k_nodes=96, k_edges=384, dtype=torch.bfloat16,
                device_w=True)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("wid,atoms", [(4, 300), (3, 400)])
def test_conv_bf16_reduced(wid, atoms):
    """bf16 storage at 128 channels: the pipelined kernels (0e+1o+2e) and the plain ones
    (0e+1o, where the bf16 pipelined kernels are not launched)."""
    w = W.WORKLOADS[wid]
    _conv_check(w, W.make_graph(w, n_atoms=atoms), tol=TOL_BF16, dtype=torch.bfloat16)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_conv_per_path_outputs_128_channels(dt):
    """One output block per path (e3j's default layout, App. E.1) on the 64k workload's irreps:
    106 output rows per node, so the forward walks each receiver's edges once per block."""
    w = W.WORKLOADS[4]
    _conv_check(w, W.make_graph(w, n_atoms=250), tol=TOL_BF16 if dt == torch.bfloat16 else TOL_F32, dtype=dt,
                per_path=True)


def test_tp_per_path_outputs_128_channels():
    w = W.Workload(94, "per-path", "tp", "128x0e+128x1o+128x2e", 3, 3, rows=777)
    _tp_check(w, None, per_path=True)


def test_conv_high_l_low_channel_reduced():
    """8x0e+8x1o+8x2e+8x3o, ~30 neighbours, 1500 atoms: every output compared."""
    w = W.WORKLOADS[5]
    _conv_check(w, W.make_graph(w, n_atoms=1500))


def test_conv_high_l_low_channel_full_size_sampled():
    """100,000 atoms, ~3.0M edges, sampled outputs."""
    w = W.WORKLOADS[5]
    _conv_check(w, W.make_graph(w), k_nodes=256, k_edges=1024)


@pytest.mark.parametrize("blocks,mul,dt", [
    ("0e+1o+2e+3o", 4, torch.float32),
    ("0e+1o+2e+3o", 16, torch.float32),
    ("0e+1o+2e+3o", 32, torch.float32),
    ("0e+1o+2e+3o", 8, torch.bfloat16),
    ("0e+1o+2e", 32, torch.float32),
    ("0e+1o", 4, torch.bfloat16),
])
def test_conv_narrow_channel_counts(blocks, mul, dt):
    """4-32 channels run the edge-slot forward (up to 8 edges of a receiver at once, their
    partial sums added across slots); a box of 400 atoms with ~30 neighbours puts receivers of
    1-8 and more slot rounds side by side, and the backward its plain kernel."""
    irreps = "+".join(f"{mul}x{b}" for b in blocks.split("+"))
    w = W.Workload(94, "narrow channels", "conv", irreps, 3, 3, n_atoms=400, degree=30.0)
    g = W.make_graph(w)
    _conv_check(w, g, tol=TOL_BF16 if dt == torch.bfloat16 else TOL_F32, dtype=dt)


def test_conv_irregular_graph_with_empty_receivers():
    w = W.Workload(94, "irregular", "conv", "16x0e+16x1o", 3, 3, n_atoms=0)
    g = random_graph(61, 500, (94, 0), empty_nodes=9)
    _conv_check(w, g)


@pytest.mark.parametrize("lmax", [0, 1, 2, 3])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_sh_backward(lmax, dt):
    """dvec = VJP of the harmonics (forces through the edge vectors)."""
    rng = np.random.default_rng(50 + lmax)
    n = 2051
    vec = (rng.standard_normal((n, 3)) * rng.uniform(0.1, 6.0, (n, 1))).astype(np.float32)
    vec[0] = 0.0
    dy = rng.standard_normal((n, (lmax + 1) ** 2)).astype(np.float32)
    dyd = to_dev(dy, dt)
    dvec = e3.sh_backward(to_dev(vec), dyd, lmax)
    torch.cuda.synchronize()
    ref = oracle.sh_grad(vec.astype(np.float64), lmax, to_np(dyd))
    # dvec scales as 1/|r|: compare |r| dvec (the gradient in the direction) so that the
    # closest pairs do not set the RMS of the whole tensor
    rn = np.linalg.norm(vec.astype(np.float64), axis=1, keepdims=True)
    assert_close(to_np(dvec) * rn, ref * rn, TOL_F32, f"|r| dvec l<={lmax}")
    assert np.all(to_np(dvec)[0] == 0.0)


def test_sh_backward_conv_edges_full_size():
    """All 2.56M edge vectors of the 64k-atom workload, 4096 sampled edges checked."""
    w = W.WORKLOADS[4]
    g = W.make_graph(w)
    vec = g.vec.astype(np.float32)
    dyd = torch.randn((g.n_edges, 16), device="cuda")
    dvec = e3.sh_backward(to_dev(vec), dyd, 3)
    torch.cuda.synchronize()
    ids = sample_ids(g.n_edges, 4096, 13)
    sel = torch.from_numpy(ids).cuda()
    ref = oracle.sh_grad(vec[ids].astype(np.float64), 3, to_np(dyd[sel]))
    rn = np.linalg.norm(vec[ids].astype(np.float64), axis=1, keepdims=True)
    assert_close(to_np(dvec[sel]) * rn, ref * rn, TOL_F32, "|r| dvec")
