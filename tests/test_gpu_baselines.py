"""The nondeterministic overhead baselines (include/det_baselines.h) run and
give results within rounding distance of the deterministic ones.  Their bits
may change from run to run, so nothing here compares bits; the number of
distinct results over repeated runs is reported by the benchmark, never
gated."""
import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


@pytest.mark.parametrize("dtype,tol", [(np.float32, 2e-6), (np.float64, 1e-14)])
def test_atomic_sum(det, dtype, tol):
    x = workloads.sum_input(n=(1 << 20) + 5, dtype=dtype)
    out = torch.empty(1, dtype=torch.float32 if dtype == np.float32 else torch.float64, device="cuda")
    det.atomic_sum(torch.from_numpy(x).cuda(), out)
    ref = float(oracle.det_sum(x))
    assert abs(float(out.item()) - ref) <= 2 * tol * float(np.abs(x.astype(np.float64)).sum())


@pytest.mark.parametrize("dtype,tol", [(np.float32, 2e-6), (np.float64, 1e-14)])
def test_atomic_scatter_add(det, dtype, tol):
    values, bins, out0 = workloads.skewed_scatter_input(n=200_000, num_bins=1000, dtype=dtype, seed=4)
    want, perm, seg = oracle.det_scatter_add(out0, bins, values)
    out = torch.from_numpy(out0.copy()).cuda()
    det.atomic_scatter_add(out, torch.from_numpy(bins).cuda(), torch.from_numpy(values).cuda())
    got = out.cpu().numpy()
    absum = np.zeros(out0.size)
    valid = (bins >= 0) & (bins < out0.size)
    np.add.at(absum, bins[valid], np.abs(values[valid].astype(np.float64)))
    assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= 2 * tol * absum + 1e-300)


@pytest.mark.parametrize("dtype,tol", [(np.float32, 2e-6), (np.float64, 1e-14)])
def test_atomic_scatter_add_rows(det, dtype, tol):
    src, idx, dst0 = workloads.rows_input(src_rows=20_000, dst_rows=2_000, row_len=64, dtype=dtype)
    idx[::7] = -1   # some skipped rows
    want, _ = oracle.det_scatter_add_rows(dst0, idx, src)
    dst = torch.from_numpy(dst0.copy()).cuda()
    prev = torch.empty(src.shape, dtype=dst.dtype, device="cuda")
    det.atomic_scatter_add_rows(dst, torch.from_numpy(idx).cuda(), torch.from_numpy(src).cuda(), prev_out=prev)
    got = dst.cpu().numpy().astype(np.float64)
    scale = np.abs(dst0).astype(np.float64) + 64.0
    assert np.all(np.abs(got - want.astype(np.float64)) <= 64 * tol * scale)
    assert not prev.cpu().numpy()[::7].any()   # skipped rows return +0.0


@pytest.mark.parametrize("dtype,rel", [(np.float32, 1e-4), (np.float64, 1e-12)])
def test_dlb_scan(det, dtype, rel):
    x = workloads.scan_input(n=3_000_017, dtype=dtype)
    want, _ = oracle.det_scan(x)
    xt = torch.from_numpy(x).cuda()
    y = torch.empty_like(xt)
    det.dlb_scan(xt, y)
    got = y.cpu().numpy().astype(np.float64)
    w = want.astype(np.float64)
    assert np.all(np.abs(got - w) <= rel * np.abs(w) + 1e-30)
