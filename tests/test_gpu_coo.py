"""Tensor product with runtime COO coefficients on the GPU (e3j App. E.1 Eq. (10)-(11),
Alg. 1) against the oracle's record loops: CG records (the CG tensor product, also against
the compile-time kernels), random records in any order with repeats, a natural-parity-only
path subset, out-of-range records, no records, and determinism."""
import numpy as np
import pytest
import torch

import message_passing_gb300 as e3
import oracle
from gpu_util import TOL_BF16, TOL_F32, assert_close, to_dev, to_np

pytestmark = pytest.mark.gpu

X2 = [(0, 1), (1, -1), (2, 1)]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda):
    e3.load()
    e3.check_device_status()
    yield
    torch.cuda.synchronize()


def _rows(R, d1, d2, P, D, mul, dtype, seed):
    r = np.random.default_rng(seed)
    x, y = r.standard_normal((R, d1, mul)), r.standard_normal((R, d2))
    w, dz = r.standard_normal((R, P, mul)) / np.sqrt(P), r.standard_normal((R, D, mul))
    return [to_dev(a.astype(np.float32), dtype) for a in (x, y, w, dz)]


def _check(recs, c, dims, mul, dtype, R=1037, seed=0):
    d1, d2, P, D = dims
    x, y, w, dz = _rows(R, d1, d2, P, D, mul, dtype, seed)
    rec_d = to_dev(np.ascontiguousarray(recs, dtype=np.int32))
    c32 = np.asarray(c, dtype=np.float32)
    c_d = to_dev(c32)
    z = e3.coo_tp_forward(rec_d, c_d, x, y, w, D)
    dx, dy, dw = e3.coo_tp_backward(rec_d, c_d, x, y, w, dz)
    assert e3.check_device_status() == 0
    xo, yo, wo, dzo = (to_np(a) for a in (x, y, w, dz))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    assert_close(to_np(z), oracle.coo_tp_forward(recs, c32, xo, yo, wo, D), tol, "z")
    for got, ref, name in zip((dx, dy, dw), oracle.coo_tp_backward(recs, c32, xo, yo, wo, dzo), ("dx", "dy", "dw")):
        assert_close(to_np(got), ref, tol, name)
    return (x, y, w, dz), (z, dx, dy, dw)


@pytest.mark.parametrize("mul", [128, 64, 32, 8])
def test_cg_records_equal_the_cg_tensor_product(mul):
    ot = oracle.table(X2, 3, 3)
    recs, c = oracle.cg_records(ot)
    (x, y, w, dz), (z, dx, dy, dw) = _check(recs, c, (ot.d1, ot.d2, ot.n_paths, ot.D), mul, torch.float32)
    t = e3.Table.create(X2, mul, 3, 3)
    assert_close(to_np(z), to_np(e3.tp_forward(t, x, y, w)), 2 * TOL_F32, "z vs compile-time kernel")
    for got, ref, name in zip((dx, dy, dw), e3.tp_backward(t, x, y, w, dz), ("dx", "dy", "dw")):
        assert_close(to_np(got), to_np(ref), 2 * TOL_F32, name + " vs compile-time kernel")


@pytest.mark.parametrize("mul,dt", [(128, torch.float32), (128, torch.bfloat16), (64, torch.float32),
                                    (16, torch.float32), (4, torch.bfloat16), (1, torch.float32)])
def test_random_records_any_order_with_repeats(mul, dt):
    r = np.random.default_rng(mul)
    d1, d2, P, D, n = 7, 5, 4, 9, 300
    recs = np.stack([r.integers(0, D, n), r.integers(0, d1, n), r.integers(0, d2, n), r.integers(0, P, n)], 1)
    recs[5] = recs[4]
    recs[D:] = recs[D:][r.permutation(n - D)]
    recs[:, 0][recs[:, 0] == 3] = 4          # output row 3 has no record: must come out zero
    (_, _, _, _), (z, _, _, _) = _check(recs, r.standard_normal(n), (d1, d2, P, D), mul, dt, R=517, seed=mul)
    assert torch.all(z[:, 3] == 0)


def test_natural_parity_only_subset():
    """Only the paths whose output parity is (-1)^l3 (e3j App. B.1), as a record subset."""
    ot = oracle.table(X2, 3, 3)
    recs, c = oracle.cg_records(ot)
    natural = np.array([p.p3 == (-1) ** p.l3 for p in ot.paths])
    keep = natural[recs[:, 3]]
    assert 0 < keep.sum() < len(keep)
    _check(recs[keep], c[keep], (ot.d1, ot.d2, ot.n_paths, ot.D), 128, torch.float32)


def test_out_of_range_record_is_skipped_and_flagged():
    r = np.random.default_rng(3)
    d1, d2, P, D = 4, 4, 2, 3
    recs = np.array([[0, 1, 2, 1], [2, 3, 0, 0], [1, 0, 1, 1]], dtype=np.int32)
    bad = np.concatenate([recs, [[1, 9, 0, 0]]]).astype(np.int32)
    c = np.array([0.5, -1.25, 2.0, 7.0], dtype=np.float32)
    x, y, w, _ = _rows(33, d1, d2, P, D, 8, torch.float32, 4)
    z = e3.coo_tp_forward(to_dev(bad), to_dev(c), x, y, w, D)
    with pytest.raises(e3.E3GBError):
        e3.check_device_status()
    assert_close(to_np(z), oracle.coo_tp_forward(recs, c[:3], to_np(x), to_np(y), to_np(w), D), TOL_F32, "z")


def test_no_records_and_determinism():
    x, y, w, dz = _rows(300, 9, 16, 24, 31, 128, torch.float32, 5)
    empty_r = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    empty_c = torch.zeros(0, dtype=torch.float32, device="cuda")
    z = e3.coo_tp_forward(empty_r, empty_c, x, y, w, 31)
    dx, dy, dw = e3.coo_tp_backward(empty_r, empty_c, x, y, w, dz)
    assert e3.check_device_status() == 0
    assert all(bool(torch.all(a == 0)) for a in (z, dx, dy, dw))
    ot = oracle.table(X2, 3, 3)
    recs, c = oracle.cg_records(ot)
    rec_d, c_d = to_dev(recs.astype(np.int32)), to_dev(c.astype(np.float32))
    a = [e3.coo_tp_backward(rec_d, c_d, x, y, w, dz) for _ in range(3)]
    for u in a[1:]:
        assert all(torch.equal(p, q) for p, q in zip(a[0], u))


@pytest.mark.parametrize("n", [8192, 8193])
def test_record_count_at_the_sorted_plan_limit(n):
    """8,192 records take the sorted-plan kernels, 8,193 the general ones: both against the
    oracle, with repeats and random order. 64 rows of every index, so that each output (z, dx,
    dy, dw) sums ~128 records (a CG list sums tens): the fp32 rounding of a sum grows with its
    length, and 1,000-term sums of random-signed terms reach the 1e-5 RMS bound by themselves."""
    r = np.random.default_rng(n)
    d1, d2, P, D = 64, 64, 64, 64
    recs = np.stack([r.integers(0, D, n), r.integers(0, d1, n), r.integers(0, d2, n), r.integers(0, P, n)], 1)
    _check(recs, r.standard_normal(n) / np.sqrt(n), (d1, d2, P, D), 16, torch.float32, R=97, seed=n)
