"""Scatter paths whose inputs start off the 16-byte boundary.

The sort's count and pass kernels bring a full tile's keys and values in by
bulk copies only from 16-byte aligned addresses; views that start one element
(or one record) in take the plain-load paths instead.  The bits must not
change: every case is compared with the CPU oracle bit for bit."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


def _offset_view(a, k=1):
    """A device copy of `a` that starts k rows into a larger buffer."""
    pad = np.zeros((k,) + a.shape[1:], a.dtype)
    full = torch.from_numpy(np.ascontiguousarray(np.concatenate([pad, a]))).cuda()
    v = full[k:]
    assert v.is_contiguous() and v.data_ptr() % 16 != 0
    return v


@pytest.mark.parametrize("m", [1024, 1 << 20])   # one-pass and two-pass sorts
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_scatter_add_offset_inputs(det, m, dtype):
    rng = np.random.default_rng(m % 97)
    n = 200_003
    values = rng.standard_normal(n).astype(dtype)
    bins = rng.integers(-7, m + 7, n).astype(np.int32)
    bins[5_000:60_000] = 11                                 # a long group
    out0 = rng.standard_normal(m).astype(dtype)
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    for bt in (0, 128):
        out = torch.from_numpy(out0.copy()).cuda()
        perm = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        seg = torch.empty(m + 1, dtype=torch.int32, device="cuda")
        det.det_scatter_add(out, _offset_view(bins), _offset_view(values), perm_out=perm, seg_offsets_out=seg,
                            block_threads=bt)
        assert np.array_equal(_bits(out.cpu().numpy()), _bits(want_out)), bt
        nvalid = int(seg[-1].item())
        assert np.array_equal(seg.cpu().numpy(), want_seg), bt
        assert np.array_equal(perm[:nvalid].cpu().numpy(), want_perm), bt


@pytest.mark.parametrize("dtype,width", [(np.float32, 3), (np.float32, 4), (np.float64, 2), (np.float32, 1)])
def test_scatter_add_vec_offset_records(det, dtype, width):
    """Records carried whole by the pass (one-pass sort, at most 16 bytes),
    from a row-major array that starts one record in."""
    rng = np.random.default_rng(width)
    n, m = 150_001, 1000
    values = rng.standard_normal((n, width)).astype(dtype)
    bins = rng.integers(-3, m + 3, n).astype(np.int32)
    bins[:40_000] = 999
    out0 = rng.standard_normal((m, width)).astype(dtype)
    want, _ = oracle.det_scatter_add_rows(out0, bins, values)
    # a record of 16 bytes stays aligned whatever row the view starts at: only its bins are offset
    shifted = values.itemsize * width % 16 != 0
    for bt in (0, 256):
        out = torch.from_numpy(out0.copy()).cuda()
        v = _offset_view(values) if shifted else torch.from_numpy(np.ascontiguousarray(values)).cuda()
        det.det_scatter_add_vec(out, _offset_view(bins), v, block_threads=bt)
        assert np.array_equal(_bits(out.cpu().numpy()), _bits(want)), bt
