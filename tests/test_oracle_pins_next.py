"""CPU pins of the oracle's scatter-sub, scatter-min/max, int32 scan, slot
allocation, the ordered row scatter, the gather and the per-segment-restart
segmented scan against facts the pages and the mathematics fix, computed here
without the oracle: integer-exact sums, numpy's grouped minimum/maximum, numpy
cumulative sums with int32 wrap-around, the pages' compaction example
(Warp "Deterministic Execution", "Pattern 2: Slot Allocation" and "Picking the
Right Mode"), and the IEEE 754-2019 minimum/maximum rules for signed zeros
and NaN written out as literal cases."""
import numpy as np
import pytest

import oracle


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


# ---------------------------------------------------------------------------
# scatter_sub: values negated and added in the fixed order of scatter_add

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_sub_integer_exact(dtype):
    rng = np.random.default_rng(11)
    n, m = 5000, 37
    values = rng.integers(-100, 100, n).astype(dtype)
    bins = rng.integers(-3, m + 3, n).astype(np.int32)   # some out of range: skipped
    out0 = rng.integers(-1000, 1000, m).astype(dtype)
    got = oracle.det_scatter_sub(out0, bins, values)
    ok = (bins >= 0) & (bins < m)
    want = out0.astype(np.int64) - np.bincount(bins[ok], weights=values[ok].astype(np.int64), minlength=m).astype(np.int64)
    assert np.array_equal(got, want.astype(dtype))


def test_sub_sign_and_untouched():
    out0 = np.array([10.0, -0.0, 7.0], np.float32)
    got = oracle.det_scatter_sub(out0, np.array([0, 0, 0], np.int32), np.array([1.0, 2.0, 3.0], np.float32))
    assert got[0] == 4.0
    assert np.array_equal(_bits(got[1:]), _bits(out0[1:]))   # bins without records keep their bits (-0.0 too)


def test_sub_negates_values_not_the_group_result():
    # (-1) + 1 is +0.0 while -(1 + (-1)) is -0.0: with old = -0.0 the two
    # readings differ, and the pages negate the values
    got = oracle.det_scatter_sub(np.array([-0.0], np.float32), np.array([0, 0], np.int32),
                                 np.array([1.0, -1.0], np.float32))
    assert got[0] == 0.0 and not np.signbit(got[0])


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_sub_equals_add_of_negated(dtype):
    # the pages define atomic_sub as "negated and added": same groups, same order
    rng = np.random.default_rng(12)
    values = rng.standard_normal(20000).astype(dtype)
    bins = rng.integers(0, 64, values.size).astype(np.int32)
    out0 = rng.standard_normal(64).astype(dtype)
    got = oracle.det_scatter_sub(out0, bins, values)
    want, _, _ = oracle.det_scatter_add(out0, bins, -values)
    assert np.array_equal(_bits(got), _bits(want))


# ---------------------------------------------------------------------------
# scatter_min / scatter_max: IEEE 754-2019 minimum / maximum, old value included

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("which", ["min", "max"])
def test_minmax_matches_numpy_grouped(dtype, which):
    rng = np.random.default_rng(13)
    n, m = 30000, 500
    values = rng.standard_normal(n).astype(dtype)
    bins = rng.integers(-10, m + 10, n).astype(np.int32)
    out0 = rng.standard_normal(m).astype(dtype)
    got = (oracle.det_scatter_min if which == "min" else oracle.det_scatter_max)(out0, bins, values)
    want = out0.copy()
    ok = (bins >= 0) & (bins < m)
    (np.minimum if which == "min" else np.maximum).at(want, bins[ok], values[ok])
    assert np.array_equal(_bits(got), _bits(want))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_minmax_signed_zero_and_nan(dtype):
    pz, nz, nan = dtype(0.0), dtype(-0.0), dtype(np.nan)
    # -0 orders below +0, whichever comes first
    out0 = np.array([pz, nz, pz, nz], dtype)
    vals = np.array([nz, pz, pz, nz], dtype)
    bins = np.array([0, 1, 2, 3], np.int32)
    mn = oracle.det_scatter_min(out0, bins, vals)
    mx = oracle.det_scatter_max(out0, bins, vals)
    assert [np.signbit(v) for v in mn] == [True, True, False, True]
    assert [np.signbit(v) for v in mx] == [False, False, False, True]
    # a NaN anywhere in a touched group (or as the old value) gives NaN
    out0 = np.array([1.0, nan, 3.0, 4.0], dtype)
    vals = np.array([2.0, 0.5, nan, -1.0, 5.0], dtype)
    bins = np.array([0, 1, 2, 2, 3], np.int32)
    mn = oracle.det_scatter_min(out0, bins, vals)
    mx = oracle.det_scatter_max(out0, bins, vals)
    assert mn[0] == 1.0 and np.isnan(mn[1]) and np.isnan(mn[2]) and mn[3] == 4.0
    assert mx[0] == 2.0 and np.isnan(mx[1]) and np.isnan(mx[2]) and mx[3] == 5.0
    # untouched entries keep their exact bits, NaN payloads included
    out0 = np.array([7.0, 7.0], dtype)
    _bits(out0)[1] = 0x7fc00123 if dtype == np.float32 else 0x7ff8000000000123
    mn = oracle.det_scatter_min(out0, np.array([0], np.int32), np.array([1.0], dtype))
    assert mn[0] == 1.0 and _bits(mn)[1] == _bits(out0)[1]


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_minmax_order_free(dtype):
    rng = np.random.default_rng(14)
    values = rng.standard_normal(4000).astype(dtype)
    values[::97] = 0.0
    values[::89] = -0.0
    values[5] = np.nan
    bins = rng.integers(0, 50, values.size).astype(np.int32)
    out0 = rng.standard_normal(50).astype(dtype)
    p = rng.permutation(values.size)
    for f in (oracle.det_scatter_min, oracle.det_scatter_max):
        a = f(out0, bins, values)
        b = f(out0, bins[p], values[p])
        assert np.array_equal(np.isnan(a), np.isnan(b))
        k = ~np.isnan(a)
        assert np.array_equal(_bits(a[k]), _bits(b[k]))


# ---------------------------------------------------------------------------
# int32 scan: modular prefix sums

def test_scan_i32_matches_cumsum_with_wrap():
    rng = np.random.default_rng(15)
    x = rng.integers(-2**31, 2**31, 100000, dtype=np.int64).astype(np.int32)
    inc, total = oracle.det_scan_i32(x)
    exc, total2 = oracle.det_scan_i32(x, exclusive=True)
    cs = np.cumsum(x.astype(np.int64))
    assert np.array_equal(inc, cs.astype(np.int32))               # int64 -> int32 wraps modulo 2^32
    assert np.array_equal(exc, (cs - x.astype(np.int64)).astype(np.int32))
    assert total == total2 == np.int64(cs[-1]).astype(np.int32)


def test_scan_i32_page_recipe():
    # offsets = exclusive scan of counts; final count = offsets[n-1] + counts[n-1]
    counts = np.array([1, 0, 1, 1, 0, 0, 1], np.int32)
    offsets, total = oracle.det_scan_i32(counts, exclusive=True)
    assert offsets.tolist() == [0, 1, 1, 2, 3, 3, 3]
    assert total == offsets[-1] + counts[-1] == 4
    assert oracle.det_scan_i32(np.zeros(0, np.int32))[1] == 0


# ---------------------------------------------------------------------------
# slot allocation

def test_slot_alloc_compaction_example():
    # compact_positive: threads with v > 0 take a slot from count[0] and write
    # v there; in thread order the result is the boolean-mask selection
    rng = np.random.default_rng(16)
    values = rng.standard_normal(10000).astype(np.float32)
    flags = (values > 0).astype(np.int32)
    slots, ctr = oracle.det_slot_alloc(np.zeros(1, np.int32), np.zeros(values.size, np.int32), count=flags)
    compacted = np.empty(int(ctr[0]), np.float32)
    compacted[slots[flags == 1]] = values[flags == 1]
    assert np.array_equal(compacted, values[values > 0])
    # the same with non-reserving threads skipped (index outside the counter array)
    idx = np.where(values > 0, 0, -1).astype(np.int32)
    slots2, ctr2 = oracle.det_slot_alloc(np.zeros(1, np.int32), idx)
    assert np.array_equal(slots2[values > 0], slots[values > 0]) and np.all(slots2[values <= 0] == -1)
    assert ctr2[0] == ctr[0] == int(np.count_nonzero(values > 0))


def test_slot_alloc_multi_counter_matches_grouped_cumsum():
    rng = np.random.default_rng(17)
    n, C = 20000, 13
    index = rng.integers(-2, C + 2, n).astype(np.int32)
    count = rng.integers(0, 5, n).astype(np.int32)
    counter0 = rng.integers(0, 1000, C).astype(np.int32)     # pre-existing nonzero counters
    slots, ctr = oracle.det_slot_alloc(counter0, index, count=count)
    want = np.full(n, -1, np.int64)
    for c in range(C):
        sel = np.flatnonzero(index == c)
        cs = np.cumsum(count[sel].astype(np.int64))
        want[sel] = counter0[c] + cs - count[sel]
    assert np.array_equal(slots, want.astype(np.int32))
    ok = (index >= 0) & (index < C)
    assert np.array_equal(ctr, counter0 + np.bincount(index[ok], weights=count[ok], minlength=C).astype(np.int32))


def test_slot_alloc_append_in_two_launches():
    # append-style multi-launch use: the second launch continues where the first stopped
    rng = np.random.default_rng(18)
    index = rng.integers(0, 4, 3000).astype(np.int32)
    s_all, c_all = oracle.det_slot_alloc(np.zeros(4, np.int32), index)
    s1, c1 = oracle.det_slot_alloc(np.zeros(4, np.int32), index[:1234])
    s2, c2 = oracle.det_slot_alloc(c1, index[1234:])
    assert np.array_equal(np.concatenate([s1, s2]), s_all) and np.array_equal(c2, c_all)


def test_slot_alloc_offset_and_empty():
    s, c = oracle.det_slot_alloc(np.array([3, 9], np.int32), np.array([5, 6, 5, 7], np.int32), index_offset=-5)
    assert s.tolist() == [3, 9, 4, -1] and c.tolist() == [5, 10]
    s, c = oracle.det_slot_alloc(np.array([3], np.int32), np.zeros(0, np.int32))
    assert s.size == 0 and c.tolist() == [3]


# ---------------------------------------------------------------------------
# ordered row scatter: contributions applied one source row at a time

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_rows_ordered_matches_numpy_add_at(dtype):
    # numpy's unbuffered add.at applies repeated indices one by one in index order
    rng = np.random.default_rng(31)
    src = rng.standard_normal((3000, 5)).astype(dtype)
    idx = rng.integers(-2, 42, 3000).astype(np.int32)
    dst0 = rng.standard_normal((40, 5)).astype(dtype)
    got, prev = oracle.det_scatter_add_rows_ordered(dst0, idx, src)
    want = dst0.copy()
    ok = (idx >= 0) & (idx < 40)
    np.add.at(want, idx[ok], src[ok])
    assert np.array_equal(_bits(got), _bits(want))
    assert not prev[~ok].any()


def test_rows_ordered_prev_is_the_running_prefix():
    # integer-valued rows: prev of the k-th contributor of r is dst0[r] + the sum of the earlier ones
    rng = np.random.default_rng(32)
    src = rng.integers(-50, 50, (5000, 3)).astype(np.float32)
    idx = rng.integers(0, 17, 5000).astype(np.int32)
    dst0 = rng.integers(-100, 100, (17, 3)).astype(np.float32)
    got, prev = oracle.det_scatter_add_rows_ordered(dst0, idx, src)
    for r in range(17):
        sel = np.flatnonzero(idx == r)
        cs = np.cumsum(src[sel].astype(np.int64), axis=0)
        assert np.array_equal(prev[sel], (dst0[r].astype(np.int64) + cs - src[sel].astype(np.int64)).astype(np.float32))
        assert np.array_equal(got[r], (dst0[r].astype(np.int64) + cs[-1]).astype(np.float32))


def test_rows_ordered_equals_default_for_distinct_rows():
    # with every destination hit at most once both readings return the plain gather
    rng = np.random.default_rng(33)
    src = rng.standard_normal((64, 4)).astype(np.float32)
    idx = rng.permutation(100)[:64].astype(np.int32)
    dst0 = rng.standard_normal((100, 4)).astype(np.float32)
    a = oracle.det_scatter_add_rows_ordered(dst0, idx, src)
    b = oracle.det_scatter_add_rows(dst0, idx, src)
    assert np.array_equal(_bits(a[0]), _bits(b[0])) and np.array_equal(_bits(a[1]), _bits(b[1]))
    assert np.array_equal(a[1], dst0[idx])


# ---------------------------------------------------------------------------
# gather (the forward of the pages' backward example)

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_gather_matches_numpy_take(dtype):
    rng = np.random.default_rng(34)
    src = rng.standard_normal((300, 7)).astype(dtype)
    idx = rng.integers(-5, 305, 2000).astype(np.int32)
    got = oracle.det_gather_rows(src, idx)
    ok = (idx >= 0) & (idx < 300)
    want = np.zeros((2000, 7), dtype)
    want[ok] = src[idx[ok]]
    assert np.array_equal(_bits(got), _bits(want))
    v = src[:, 0].copy()
    assert np.array_equal(_bits(oracle.det_gather_rows(v, idx)), _bits(want[:, 0]))
    assert np.array_equal(oracle.det_gather_rows(src, idx + 3, row_offset=-3), got)


# ---------------------------------------------------------------------------
# per-segment-restart segmented scan (flag 4): each segment scanned alone

R = oracle.SCAN_SEGMENT_RESTART


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_restart_ones_closed_form(dtype, flags):
    # x = 1: inclusive = 1-based position in the segment, exclusive = 0-based;
    # reverse counts from the segment's end; segments span several chunks
    C = oracle.scan_chunk_elems(dtype)
    lens = [5, 0, 3 * C + 17, 1, C, 40 * C + 3]          # the last one spans anchor intervals
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = np.ones(int(off[-1]), dtype)
    y = oracle.det_segmented_scan(x, off, flags | R)
    for s_, L in enumerate(lens):
        p = np.arange(L, dtype=np.float64)
        if flags & 2:
            p = p[::-1]
        want = p + (0 if flags & 1 else 1)
        assert np.array_equal(y[off[s_]:off[s_ + 1]].astype(np.float64), want)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_restart_short_segments_are_sequential(dtype):
    # a segment no longer than one lane is a single lane fold: numpy's cumsum order
    E = oracle.scan_lane_elems(dtype)
    rng = np.random.default_rng(35)
    lens = rng.integers(1, E + 1, 400)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = rng.lognormal(0, 1, int(off[-1])).astype(dtype)
    y = oracle.det_segmented_scan(x, off, R)
    for s_ in range(lens.size):
        seg = x[off[s_]:off[s_ + 1]]
        assert np.array_equal(_bits(y[off[s_]:off[s_ + 1]]), _bits(np.cumsum(seg, dtype=dtype)))


def test_restart_differs_from_the_global_grid_reading():
    # a segment starting at 5 (f32 lanes hold 32 elements): values at segment
    # positions 0, 30, 60, 90.  Alone, 0 and 30 share lane 0 and position 95 is
    # ((v0 + v30) + v60) + v90; on the global grid they land in lanes 0, 1, 2, 2
    # and position 95 (global 100, lane 3) is v0 + (v30 + (v60 + v90)).
    x = np.full(128, -0.0, np.float32)
    x[5 + np.array([0, 30, 60, 90])] = [2.0**24, 1.0, 1.0, 1.0]
    off = np.array([0, 5, 128], np.int64)
    a = oracle.det_segmented_scan(x, off, R)
    b = oracle.det_segmented_scan(x, off)
    assert a[5 + 95] == np.float32(2.0**24)              # (((2^24 + 1) + 1) + 1) rounds to 2^24 each time
    assert b[5 + 95] == np.float32(2.0**24 + 4)          # 2^24 + 3 rounds to 2^24 + 4
    one = oracle.det_scan(x[:5])[0], oracle.det_scan(x[5:])[0]
    assert np.array_equal(_bits(a), _bits(np.concatenate(one)))


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_restart_single_segment_is_the_full_scan(flags):
    rng = np.random.default_rng(36)
    x = rng.lognormal(0, 1, 100_003).astype(np.float32)
    off = np.array([0, x.size], np.int64)
    assert np.array_equal(_bits(oracle.det_segmented_scan(x, off, flags | R)),
                          _bits(oracle.det_scan(x, flags)[0]))
