"""GPU parity of scatter-sub, scatter-min/max, the int32 scan and slot
allocation against the CPU oracle, bit for bit, through the C ABI."""
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


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


def _same_float(got, want):
    """Bitwise equality; NaN positions must agree (payloads are not promised)."""
    got, want = np.asarray(got), np.asarray(want)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    k = ~np.isnan(want)
    assert np.array_equal(_bits(got[k]), _bits(want[k]))


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ---------------------------------------------------------------------------
# scatter_sub

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bt", [128, 256, 1024])
def test_scatter_sub_skewed(det, dtype, bt):
    values, bins, out0 = workloads.skewed_scatter_input(n=300_017, num_bins=5000, dtype=dtype, seed=21)
    want = oracle.det_scatter_sub(out0, bins, values)
    out = _cuda(out0.copy())
    det.det_scatter_sub(out, _cuda(bins), _cuda(values), block_threads=bt)
    _same_float(out.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_scatter_sub_long_bins_and_perm(det, dtype):
    # one bin with 2^20 records (block trees + last-block merge), plus a few small ones
    values, bins, out0 = workloads.scatter_input(n=(1 << 20) + 333, num_bins=7, dtype=dtype, all_in_bin0=False)
    bins[: 1 << 20] = 3
    want = oracle.det_scatter_sub(out0, bins, values)
    _, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    out = _cuda(out0.copy())
    perm = torch.empty(bins.size, dtype=torch.int32, device="cuda")
    seg = torch.empty(out0.size + 1, dtype=torch.int32, device="cuda")
    det.det_scatter_sub(out, _cuda(bins), _cuda(values), perm_out=perm, seg_offsets_out=seg)
    _same_float(out.cpu().numpy(), want)
    assert np.array_equal(perm.cpu().numpy()[: want_perm.size], want_perm)
    assert np.array_equal(seg.cpu().numpy(), want_seg)


def test_scatter_sub_negates_the_values(det):
    # (-1) + 1 = +0.0, so -0.0 - group([1, -1]) is +0.0
    out0 = np.array([-0.0, -0.0], np.float32)
    bins = np.array([0, 0, 1], np.int32)
    values = np.array([1.0, -1.0, 0.0], np.float32)
    want = oracle.det_scatter_sub(out0, bins, values)
    out = _cuda(out0.copy())
    det.det_scatter_sub(out, _cuda(bins), _cuda(values))
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(want))


# ---------------------------------------------------------------------------
# scatter_min / scatter_max

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("which", ["min", "max"])
@pytest.mark.parametrize("m", [1000, 8192, 1 << 20])   # shared-memory keys up to 8,192 bins, global beyond
def test_scatter_minmax(det, dtype, which, m):
    values, bins, out0 = workloads.skewed_scatter_input(n=400_009, num_bins=m, dtype=dtype, seed=22)
    values[::1013] = 0.0
    values[::1019] = -0.0
    out0[::7] = -0.0
    f_or = oracle.det_scatter_min if which == "min" else oracle.det_scatter_max
    f_det = det.det_scatter_min if which == "min" else det.det_scatter_max
    want = f_or(out0, bins, values)
    for bt in (128, 256):
        out = _cuda(out0.copy())
        f_det(out, _cuda(bins), _cuda(values), block_threads=bt)
        _same_float(out.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_scatter_minmax_nan_zero_hot_and_untouched(det, dtype):
    n = 100_000
    rng = np.random.default_rng(23)
    values = rng.standard_normal(n).astype(dtype)
    bins = np.zeros(n, np.int32)                  # one hot bin
    bins[1::3] = 1
    bins[2::3] = rng.integers(2, 6, bins[2::3].size)
    values[777] = np.nan                          # bin 1's group holds a NaN
    bins[777] = 1
    out0 = np.array([5.0, 0.0, -0.0, np.nan, 1e30, 7.0, 9.0], dtype)
    _bits(out0)[6] = 0x7fc00123 if dtype == np.float32 else 0x7ff8000000000123   # untouched NaN keeps its payload
    for fo, fd in ((oracle.det_scatter_min, det.det_scatter_min), (oracle.det_scatter_max, det.det_scatter_max)):
        want = fo(out0, bins, values)
        out = _cuda(out0.copy())
        fd(out, _cuda(bins), _cuda(values))
        got = out.cpu().numpy()
        _same_float(got, want)
        assert _bits(got)[6] == _bits(out0)[6]


# ---------------------------------------------------------------------------
# int32 scan

@pytest.mark.parametrize("n", [0, 1, 4095, 4096, 4097, 3 * 4096 + 17, 1_000_003])
@pytest.mark.parametrize("exclusive", [False, True])
def test_scan_i32(det, n, exclusive):
    rng = np.random.default_rng(24)
    x = rng.integers(-2**31, 2**31, n, dtype=np.int64).astype(np.int32)
    want, want_total = oracle.det_scan_i32(x, exclusive=exclusive)
    xt = _cuda(x)
    total = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = det.det_scan_i32(xt, exclusive=exclusive, total_out=total)
    assert np.array_equal(y.cpu().numpy(), want)
    assert int(total.item()) == want_total
    # in place, and from an offset (unaligned) view
    det.det_scan_i32(xt, xt, exclusive=exclusive)
    assert np.array_equal(xt.cpu().numpy(), want)
    if n > 3:
        x2 = _cuda(x)[1:]
        w2, _ = oracle.det_scan_i32(x[1:], exclusive=exclusive)
        assert np.array_equal(det.det_scan_i32(x2, exclusive=exclusive).cpu().numpy(), w2)


# ---------------------------------------------------------------------------
# slot allocation

@pytest.mark.parametrize("C", [1, 13, 5000, 1 << 20])   # shared / global segment starts; 1 and 2 sort passes
@pytest.mark.parametrize("with_count", [False, True])
def test_slot_alloc(det, C, with_count):
    rng = np.random.default_rng(25 + C)
    n = 300_001
    index = rng.integers(-3, C + 3, n).astype(np.int32)
    count = rng.integers(0, 6, n).astype(np.int32) if with_count else None
    counter0 = rng.integers(0, 1000, C).astype(np.int32)
    want_slots, want_ctr = oracle.det_slot_alloc(counter0, index, count=count)
    for bt in (128, 256, 1024):
        ctr = _cuda(counter0.copy())
        slots = det.det_slot_alloc(ctr, _cuda(index), count=None if count is None else _cuda(count), block_threads=bt)
        assert np.array_equal(slots.cpu().numpy(), want_slots)
        assert np.array_equal(ctr.cpu().numpy(), want_ctr)


def test_slot_alloc_compaction_and_append(det):
    # the pages' compact_positive in two launches on one counter
    rng = np.random.default_rng(26)
    values = rng.standard_normal(200_003).astype(np.float32)
    idx = np.where(values > 0, 0, -1).astype(np.int32)
    ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
    s1 = det.det_slot_alloc(ctr, _cuda(idx[:77_777]))
    s2 = det.det_slot_alloc(ctr, _cuda(idx[77_777:]))
    slots = np.concatenate([s1.cpu().numpy(), s2.cpu().numpy()])
    want_slots, want_ctr = oracle.det_slot_alloc(np.zeros(1, np.int32), idx)
    assert np.array_equal(slots, want_slots) and int(ctr.item()) == int(want_ctr[0])
    compacted = np.empty(int(want_ctr[0]), np.float32)
    compacted[slots[slots >= 0]] = values[slots >= 0]
    assert np.array_equal(compacted, values[values > 0])


def test_slot_alloc_offset_and_empty(det):
    ctr = _cuda(np.array([3, 9], np.int32))
    s = det.det_slot_alloc(ctr, _cuda(np.array([5, 6, 5, 7], np.int32)), index_offset=-5)
    assert s.cpu().numpy().tolist() == [3, 9, 4, -1] and ctr.cpu().numpy().tolist() == [5, 10]
    s = det.det_slot_alloc(ctr, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert s.numel() == 0 and ctr.cpu().numpy().tolist() == [5, 10]


# ---------------------------------------------------------------------------
# the benchmark's configurations, full size

@pytest.mark.parametrize("op", ["sub", "min", "max"])
def test_next_ops_at_bench_size(det, op):
    values, bins, out0 = workloads.scatter_input(dtype=np.float32)
    f_or = {"sub": oracle.det_scatter_sub, "min": oracle.det_scatter_min, "max": oracle.det_scatter_max}[op]
    f_det = {"sub": det.det_scatter_sub, "min": det.det_scatter_min, "max": det.det_scatter_max}[op]
    want = f_or(out0, bins, values)
    out = _cuda(out0.copy())
    f_det(out, _cuda(bins), _cuda(values))
    _same_float(out.cpu().numpy(), want)


def test_slot_alloc_at_bench_size(det):
    values, _, _ = workloads.scatter_input(dtype=np.float32)
    idx = np.where(values > 0, 0, -1).astype(np.int32)
    want_slots, want_ctr = oracle.det_slot_alloc(np.zeros(1, np.int32), idx)
    ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = det.det_slot_alloc(ctr, _cuda(idx))
    assert np.array_equal(slots.cpu().numpy(), want_slots) and int(ctr.item()) == int(want_ctr[0])


# ---------------------------------------------------------------------------
# composite values and the ordered row scatter

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("width", [1, 3, 4, 9])
def test_scatter_add_vec(det, dtype, width):
    rng = np.random.default_rng(40 + width)
    n, m = 300_007, 777
    values = rng.standard_normal((n, width)).astype(dtype)
    bins = rng.integers(-5, m + 5, n).astype(np.int32)
    bins[:100_000] = 3                                     # one long group: block trees + merge
    out0 = rng.standard_normal((m, width)).astype(dtype)
    want, _ = oracle.det_scatter_add_rows(out0, bins, values)
    for bt in (128, 256, 1024):
        out = _cuda(out0.copy())
        det.det_scatter_add_vec(out, _cuda(bins), _cuda(values), block_threads=bt)
        assert np.array_equal(_bits(out.cpu().numpy()), _bits(want))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("W", [1, 3, 64, 100])
def test_scatter_add_rows_ordered(det, dtype, W):
    rng = np.random.default_rng(50 + W)
    M, R = 40_003, 1_500
    src = rng.standard_normal((M, W)).astype(dtype)
    idx = rng.integers(-3, R + 3, M).astype(np.int32)
    idx[:3000] = 7                                         # a long run on one destination
    dst0 = rng.standard_normal((R, W)).astype(dtype)
    want, want_prev = oracle.det_scatter_add_rows_ordered(dst0, idx, src)
    for bt in (128, 256):
        dst = _cuda(dst0.copy())
        prev = torch.empty(src.shape, dtype=dst.dtype, device="cuda")
        det.det_scatter_add_rows(dst, _cuda(idx), _cuda(src), prev_out=prev, ordered=True, block_threads=bt)
        assert np.array_equal(_bits(dst.cpu().numpy()), _bits(want))
        assert np.array_equal(_bits(prev.cpu().numpy()), _bits(want_prev))


def test_rows_ordered_at_bench_size(det):
    src, idx, dst0 = workloads.rows_input(dtype=np.float32)
    want, want_prev = oracle.det_scatter_add_rows_ordered(dst0, idx, src)
    dst = _cuda(dst0.copy())
    prev = torch.empty(src.shape, dtype=dst.dtype, device="cuda")
    det.det_scatter_add_rows(dst, _cuda(idx), _cuda(src), prev_out=prev, ordered=True)
    assert np.array_equal(_bits(dst.cpu().numpy()), _bits(want))
    assert np.array_equal(_bits(prev.cpu().numpy()), _bits(want_prev))


# ---------------------------------------------------------------------------
# per-segment-restart segmented scan

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_segmented_scan_restart(det, dtype, flags):
    C = oracle.scan_chunk_elems(dtype)
    rng = np.random.default_rng(90 + flags)
    geo = list(rng.geometric(1 / 4096, 300))
    lens = [0, 1, 7, 33, C - 1, C, C + 1, 0, 40 * C + 3] + geo + [5]   # empty, lane-sized, chunk edges, anchors
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = rng.lognormal(0, 1, int(off[-1])).astype(dtype)
    want = oracle.det_segmented_scan(x, off, flags | oracle.SCAN_SEGMENT_RESTART)
    xt = _cuda(x)
    ot = _cuda(off)
    got = det.det_segmented_scan(xt, ot, flags=flags | det.SCAN_SEGMENT_RESTART)
    assert np.array_equal(_bits(got.cpu().numpy()), _bits(want))
    det.det_segmented_scan(xt, ot, xt, flags=flags | det.SCAN_SEGMENT_RESTART)   # in place
    assert np.array_equal(_bits(xt.cpu().numpy()), _bits(want))


def test_segmented_scan_restart_bench_size(det):
    x = workloads.scan_input(n=workloads.SCAN_N, dtype=np.float32)
    off = workloads.segment_offsets(x.size)
    want = oracle.det_segmented_scan(x, off, oracle.SCAN_SEGMENT_RESTART)
    got = det.det_segmented_scan(_cuda(x), _cuda(off), flags=det.SCAN_SEGMENT_RESTART)
    assert np.array_equal(_bits(got.cpu().numpy()), _bits(want))
