"""Pins for the CPU oracle: each check compares the oracle with something that
is not the oracle -- values the pages print, exact integer arithmetic, brute
force over every bracketing of a few leaves, hand-derived brackets of the
frozen association order, library routines (stable argsort, bincount), and an
exactly rounded reference within the a-priori error bound.

A plausible slip in the oracle (a dropped term, a wrong pairing, a wrong lane
or chunk index, a transposed operand of the segmented operator) fails at least
one of these.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

F32, F64 = np.float32, np.float64


# --------------------------------------------------------------------------
# helpers: bracket trees over leaves, evaluated in a given precision


def all_trees(leaves):
    """Every full binary bracketing of the ordered leaves (Catalan many)."""
    if len(leaves) == 1:
        return [leaves[0]]
    out = []
    for k in range(1, len(leaves)):
        for left in all_trees(leaves[:k]):
            for right in all_trees(leaves[k:]):
                out.append((left, right))
    return out


def evaluate(tree, val, dtype):
    if isinstance(tree, tuple):
        return dtype(evaluate(tree[0], val, dtype) + evaluate(tree[1], val, dtype))
    return dtype(val[tree])


def parse(expr):
    """'((a+b)+c)' -> nested tuples of leaf names; '+' binds as written."""
    pos = 0

    def node():
        nonlocal pos
        if expr[pos] == "(":
            pos += 1
            left = node()
            assert expr[pos] == "+"
            pos += 1
            right = node()
            assert expr[pos] == ")"
            pos += 1
            return (left, right)
        start = pos
        while pos < len(expr) and expr[pos] not in "+()":
            pos += 1
        return expr[start:pos]

    tree = node()
    assert pos == len(expr), expr
    return tree


def canonical(tree, order):
    """The same bracket with each node's children swapped so that the leaves
    read in ``order`` (IEEE addition is commutative, so the bits agree)."""
    rank = {nm: i for i, nm in enumerate(order)}
    if not isinstance(tree, tuple):
        return tree
    a, b = canonical(tree[0], order), canonical(tree[1], order)
    if min(rank[x] for x in leaves_of(a)) > min(rank[x] for x in leaves_of(b)):
        a, b = b, a
    return (a, b)


def leaves_of(tree):
    return leaves_of(tree[0]) + leaves_of(tree[1]) if isinstance(tree, tuple) else [tree]


def distinguishing_values(names, dtype, rng, target, tries=40000):
    """Values of the ordered leaves for which the bracketing ``target`` gives
    bits that no other bracketing of the same leaves gives."""
    trees = all_trees(list(names))
    for t in range(tries):
        if t % 2:
            v = rng.standard_normal(len(names)) * 2.0 ** rng.uniform(-3, 3, len(names))
        else:
            v = (rng.choice([-1.0, 1.0], len(names)) * rng.uniform(1.0, 2.0, len(names))
                 * 2.0 ** rng.integers(-3, 4, len(names)).astype(np.float64))
        vals = {nm: dtype(x) for nm, x in zip(names, v)}
        want = np.array(evaluate(target, vals, dtype), dtype=dtype).tobytes()
        hits = sum(np.array(evaluate(tr, vals, dtype), dtype=dtype).tobytes() == want for tr in trees)
        if hits == 1:
            return vals
    raise RuntimeError("no distinguishing values found")


def same_bits(a, b):
    a = np.asarray(a)
    b = np.asarray(b, dtype=a.dtype)
    return a.tobytes() == b.tobytes()


# --------------------------------------------------------------------------
# det_sum: the canonical pairwise tree


# Hand-derived from the definition (pad to the next power of two with absent
# terms, pair (2j, 2j+1) level by level).
PT_BRACKETS = {
    2: "(0+1)",
    3: "((0+1)+2)",
    4: "((0+1)+(2+3))",
    5: "(((0+1)+(2+3))+4)",
    6: "(((0+1)+(2+3))+(4+5))",
    7: "(((0+1)+(2+3))+((4+5)+6))",
}


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("n", sorted(PT_BRACKETS))
def test_sum_brute_force_bracketing(n, dtype):
    rng = np.random.default_rng(100 + n)
    names = [str(i) for i in range(n)]
    vals = distinguishing_values(names, dtype, rng, parse(PT_BRACKETS[n]))
    x = np.array([vals[nm] for nm in names], dtype=dtype)
    got = oracle.det_sum(x)
    want = evaluate(parse(PT_BRACKETS[n]), vals, dtype)
    assert same_bits(got, want)
    # and no other bracketing of these leaves gives those bits
    matches = [t for t in all_trees(names) if same_bits(evaluate(t, vals, dtype), got)]
    assert matches == [parse(PT_BRACKETS[n])]


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("n,positions,bracket", [
    # [0,4)->x3, [4,8)->x4+x7, [8,16)->x8
    (16, [3, 4, 7, 8], "((3+(4+7))+8)"),
    # x5,x6 meet at level 2, x1000 joins at level 10, x1025 at level 11
    (4096, [5, 6, 1000, 1025], "(((5+6)+1000)+1025)"),
    # odd length: 9 -> padded to 16; (0,1) is a level-1 pair, x7 joins at
    # level 3, x8 is alone until the root
    (9, [0, 1, 7, 8], "(((0+1)+7)+8)"),
    # x2 and x3 are a level-1 pair; x4 joins at level 3; x1048575 at the root
    (1 << 20, [2, 3, 4, (1 << 20) - 1], "(((2+3)+4)+1048575)"),
])
def test_sum_sparse_fingerprint(n, positions, bracket, dtype):
    """Nonzeros in a sea of -0.0 expose the tree restricted to those leaves."""
    rng = np.random.default_rng(7)
    names = [str(p) for p in positions]
    vals = distinguishing_values(names, dtype, rng, canonical(parse(bracket), names))
    x = np.full(n, -0.0, dtype=dtype)
    for p in positions:
        x[p] = vals[str(p)]
    got = oracle.det_sum(x)
    assert same_bits(got, evaluate(parse(bracket), vals, dtype))


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 31, 32, 33, 1000, 4096, 65537])
def test_sum_integer_exact(n, dtype):
    rng = np.random.default_rng(n)
    ints = rng.integers(-100, 101, n)
    got = oracle.det_sum(ints.astype(dtype))
    assert got == int(ints.sum())


def test_sum_quickstart_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "quickstart_ones.json")))
    for dtype in (F32, F64):
        got = oracle.det_sum(np.full(g["n"], g["value"], dtype=dtype))
        assert got == g["expected_out"][0]


@pytest.mark.parametrize("dtype", [F32, F64])
def test_sum_signed_zeros(dtype):
    assert same_bits(oracle.det_sum(np.zeros(0, dtype)), dtype(0.0))
    assert same_bits(oracle.det_sum(np.full(7, -0.0, dtype)), dtype(-0.0))
    assert same_bits(oracle.det_sum(np.array([-0.0, 0.0, -0.0], dtype)), dtype(0.0))


@pytest.mark.parametrize("dtype,bound", [(F32, 2e-6), (F64, 1e-14)])
@pytest.mark.parametrize("dist", ["uniform", "normal", "lognormal"])
def test_sum_error_bound_vs_exact(dtype, bound, dist):
    n = 1 << 20
    rng = np.random.default_rng(11)
    x = {"uniform": lambda: rng.uniform(0, 12, n), "normal": lambda: rng.standard_normal(n),
         "lognormal": lambda: rng.lognormal(0, 1, n)}[dist]().astype(dtype)
    exact = math.fsum(x.astype(np.float64))   # exactly rounded (Shewchuk)
    got = float(oracle.det_sum(x))
    abs_sum = math.fsum(np.abs(x.astype(np.float64)))
    u = 2.0 ** -24 if dtype == F32 else 2.0 ** -53
    depth = math.ceil(math.log2(n))
    assert abs(got - exact) <= depth * u / (1 - depth * u) * abs_sum
    assert abs(got - exact) <= bound * abs_sum


def test_fsum_is_exactly_rounded():
    from fractions import Fraction
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(2000) * 2.0 ** rng.integers(-30, 30, 2000)).astype(np.float64)
    exact = sum(Fraction(float(v)) for v in x)
    assert math.fsum(x) == float(exact)


# --------------------------------------------------------------------------
# det_scatter_add


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_quickstart_golden(golden_dir, dtype):
    g = json.load(open(os.path.join(golden_dir, "quickstart_ones.json")))
    values = np.full(g["n"], g["value"], dtype=dtype)
    bins = np.full(g["n"], g["bin"], dtype=np.int32)
    out, perm, seg = oracle.det_scatter_add(np.zeros(g["out_len"], dtype), bins, values)
    assert out.tolist() == g["expected_out"]
    assert perm.tolist() == list(range(g["n"]))
    assert seg.tolist() == [0, g["n"]]


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_perm_and_offsets_match_library_sort(dtype):
    rng = np.random.default_rng(5)
    n, m = 50000, 300
    bins = rng.integers(-20, m + 20, n, dtype=np.int32)
    values = rng.standard_normal(n).astype(dtype)
    out, perm, seg = oracle.det_scatter_add(np.zeros(m, dtype), bins, values)
    valid = (bins >= 0) & (bins < m)
    idx = np.nonzero(valid)[0]
    want_perm = idx[np.argsort(bins[idx], kind="stable")]
    assert np.array_equal(perm, want_perm)
    want_seg = np.concatenate([[0], np.cumsum(np.bincount(bins[idx], minlength=m))])
    assert np.array_equal(seg, want_seg)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_integer_exact_and_reduce_by_bin(dtype):
    """Integer-valued records: every order is exact, so the result must equal
    the Warp guide's manual reduce_by_bin ("Writing Manual Deterministic
    Code": one output per bin, inputs visited in index order) and bincount."""
    rng = np.random.default_rng(9)
    n, m = 3000, 17
    bins = rng.integers(-2, m + 2, n, dtype=np.int32)
    values = rng.integers(-50, 51, n).astype(dtype)
    out0 = rng.integers(-5, 6, m).astype(dtype)
    out, _, _ = oracle.det_scatter_add(out0, bins, values)
    manual = out0.astype(np.float64).copy()
    for b in range(m):
        total = 0.0
        for i in range(n):
            if bins[i] == b:
                total += float(values[i])
        manual[b] += total
    assert np.array_equal(out.astype(np.float64), manual)
    valid = (bins >= 0) & (bins < m)
    want = out0.astype(np.int64) + np.bincount(bins[valid], weights=values[valid].astype(np.int64),
                                              minlength=m).astype(np.int64)
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_all_in_one_bin_equals_sum(dtype):
    """All records in bin 0: out[0] == old + PT(values), i.e. det_sum's bits."""
    values, bins, out0 = workloads.scatter_input(n=100003, num_bins=4, dtype=dtype, all_in_bin0=True)
    out, _, _ = oracle.det_scatter_add(out0, bins, values)
    assert same_bits(out[0], dtype(dtype(0.0) + oracle.det_sum(values)))
    assert same_bits(out[1:], out0[1:])


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_group_fingerprint(dtype):
    """Bin 1's records sit at interleaved input positions; the tree runs over
    their rank inside the bin (0..5), padded to 8:
    ((r0+r1)+(r2+r3))+(r4+r5), then old + that."""
    rng = np.random.default_rng(21)
    names = ["r0", "r1", "r2", "r3", "r4", "r5"]
    vals = distinguishing_values(names, dtype, rng, parse("(((r0+r1)+(r2+r3))+(r4+r5))"))
    old = dtype(rng.standard_normal())
    bins = np.array([0, 1, 2, 1, 1, 0, 1, 1, 3, 1], dtype=np.int32)
    values = rng.standard_normal(bins.size).astype(dtype)
    pos = np.nonzero(bins == 1)[0]
    for nm, p in zip(names, pos):
        values[p] = vals[nm]
    out0 = np.zeros(4, dtype)
    out0[1] = old
    out, _, _ = oracle.det_scatter_add(out0, bins, values)
    group = evaluate(parse("(((r0+r1)+(r2+r3))+(r4+r5))"), vals, dtype)
    assert same_bits(out[1], dtype(old + group))


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scatter_skips_out_of_range_and_keeps_untouched_bits(dtype):
    bins = np.array([-1, 5, 2, -2147483648, 2147483647, 2], dtype=np.int32)
    values = np.array([1, 2, 3, 4, 5, 6], dtype=dtype)
    out0 = np.array([-0.0, 7.0, 0.5, -0.0, 1.0], dtype=dtype)
    out, perm, seg = oracle.det_scatter_add(out0, bins, values)
    assert same_bits(out, np.array([-0.0, 7.0, 9.5, -0.0, 1.0], dtype=dtype))
    assert perm.tolist() == [2, 5]
    assert seg.tolist() == [0, 0, 0, 2, 2, 2]


@pytest.mark.parametrize("dtype,u", [(F32, 2.0 ** -24), (F64, 2.0 ** -53)])
def test_scatter_error_bound(dtype, u):
    values, bins, out0 = workloads.skewed_scatter_input(n=1 << 18, num_bins=1 << 10, dtype=dtype)
    out, perm, seg = oracle.det_scatter_add(out0, bins, values)
    for b in range(0, 1 << 10, 37):
        grp = values[perm[seg[b]:seg[b + 1]]].astype(np.float64)
        if grp.size == 0:
            continue
        exact = math.fsum(grp)
        d = math.ceil(math.log2(grp.size)) + 1 if grp.size > 1 else 1
        bound = d * u / (1 - d * u) * math.fsum(np.abs(grp))
        assert abs(float(out[b]) - exact) <= bound
        assert abs(float(out[b]) - exact) <= (2e-6 if dtype == F32 else 1e-14) * math.fsum(np.abs(grp))


# --------------------------------------------------------------------------
# det_scatter_add_rows


@pytest.mark.parametrize("dtype", [F32, F64])
def test_rows_tile_example_golden(golden_dir, dtype):
    g = json.load(open(os.path.join(golden_dir, "tile_atomic_add_indexed_example.json")))
    dst, prev = oracle.det_scatter_add_rows(np.array(g["y"], dtype), np.array(g["indices"], np.int32),
                                            np.array(g["x"], dtype))
    assert dst.tolist() == g["expected_y"]
    assert prev.tolist() == g["expected_previous"]


@pytest.mark.parametrize("dtype", [F32, F64])
def test_rows_width_one_equals_scatter(dtype):
    rng = np.random.default_rng(4)
    M, R = 5000, 64
    src = rng.standard_normal((M, 1)).astype(dtype)
    idx = rng.integers(-3, R + 3, M, dtype=np.int32)
    dst0 = rng.standard_normal((R, 1)).astype(dtype)
    dst, _ = oracle.det_scatter_add_rows(dst0, idx, src)
    out, _, _ = oracle.det_scatter_add(dst0[:, 0], idx, src[:, 0])
    assert same_bits(dst[:, 0], out)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_rows_each_column_is_a_scatter_and_prev_is_a_gather(dtype):
    rng = np.random.default_rng(6)
    M, R, W = 4000, 300, 5
    src = rng.standard_normal((M, W)).astype(dtype)
    idx = rng.integers(-10, R + 10, M, dtype=np.int32)
    dst0 = rng.standard_normal((R, W)).astype(dtype)
    off = 3
    dst, prev = oracle.det_scatter_add_rows(dst0, idx, src, row_offset=off)
    for j in range(W):
        out, _, _ = oracle.det_scatter_add(dst0[:, j], idx + off, src[:, j])
        assert same_bits(dst[:, j], out)
    r = idx.astype(np.int64) + off
    valid = (r >= 0) & (r < R)
    assert same_bits(prev[valid], dst0[r[valid]])
    assert same_bits(prev[~valid], np.zeros_like(prev[~valid]))


@pytest.mark.parametrize("dtype", [F32, F64])
def test_rows_repeated_integer_exact(dtype):
    rng = np.random.default_rng(8)
    M, R, W = 2000, 7, 3
    src = rng.integers(-9, 10, (M, W)).astype(dtype)
    idx = rng.integers(0, R, M, dtype=np.int32)
    dst0 = rng.integers(-9, 10, (R, W)).astype(dtype)
    dst, prev = oracle.det_scatter_add_rows(dst0, idx, src)
    want = dst0.astype(np.int64).copy()
    np.add.at(want, idx, src.astype(np.int64))
    assert np.array_equal(dst.astype(np.int64), want)
    assert same_bits(prev, dst0[idx])


# --------------------------------------------------------------------------
# det_scan


def scan_geometry(dtype):
    return oracle.scan_lane_elems(dtype), oracle.scan_chunk_elems(dtype)


def test_scan_geometry_is_the_frozen_one():
    assert scan_geometry(F32) == (32, 32 * 32 * 32)
    assert scan_geometry(F64) == (16, 32 * 32 * 16)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_ones_closed_form(dtype):
    _, C = scan_geometry(dtype)
    n = 2 * 32 * C + 3 * C + 12345          # spans two anchor intervals and a ragged tail
    x = np.ones(n, dtype)
    i = np.arange(n, dtype=np.float64)
    y, total = oracle.det_scan(x, oracle.SCAN_INCLUSIVE)
    assert np.array_equal(y.astype(np.float64), i + 1) and total == n
    y, _ = oracle.det_scan(x, oracle.SCAN_EXCLUSIVE)
    assert np.array_equal(y.astype(np.float64), i)
    y, total = oracle.det_scan(x, oracle.SCAN_INCLUSIVE | oracle.SCAN_REVERSE)
    assert np.array_equal(y.astype(np.float64), n - i) and total == n
    y, _ = oracle.det_scan(x, oracle.SCAN_EXCLUSIVE | oracle.SCAN_REVERSE)
    assert np.array_equal(y.astype(np.float64), n - 1 - i)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_integer_exact(dtype):
    _, C = scan_geometry(dtype)
    rng = np.random.default_rng(12)
    n = 33 * C + 77
    ints = rng.integers(-3, 4, n)
    y, total = oracle.det_scan(ints.astype(dtype))
    assert np.array_equal(y.astype(np.int64), np.cumsum(ints)) and total == ints.sum()


def _fingerprint_case(dtype, C, E, spots, query, bracket, seed):
    """spots: {leaf name: position}; query: output index; bracket: expected."""
    rng = np.random.default_rng(seed)
    order = sorted(spots, key=lambda nm: spots[nm])
    vals = distinguishing_values(order, dtype, rng, canonical(parse(bracket), order))
    n = max(spots.values()) + 1 + E
    x = np.full(n, -0.0, dtype)
    for nm, p in spots.items():
        x[p] = vals[nm]
    y, _ = oracle.det_scan(x)
    assert same_bits(y[query], evaluate(parse(bracket), vals, dtype)), (bracket, y[query])
    hits = [t for t in all_trees(order) if same_bits(evaluate(t, vals, dtype), y[query])]
    assert len(hits) == 1


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_within_chunk(dtype):
    """Lane 0 and lane 1 of warp 0, then warp 1: the warp-1 carry is the
    lane-Kogge-Stone total of warp 0, (a+b); c is then folded in."""
    E, C = scan_geometry(dtype)
    spots = {"a": 0, "b": E + 3, "c": 32 * E + 5}
    _fingerprint_case(dtype, C, E, spots, 32 * E + 5, "((a+b)+c)", 1)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_lane_kogge_stone(dtype):
    """Lanes 0,1,2,3 of warp 0 hold a,b,c,d; warp 1's carry is K[31] of the
    lane Kogge-Stone: step r=0 gives (a+b),(b+c),(c+d); r=1 gives
    (a+b)+(c+d) at lane 3; then e in warp 1 is folded in."""
    E, C = scan_geometry(dtype)
    spots = {"a": 0, "b": E, "c": 2 * E, "d": 3 * E, "e": 32 * E}
    _fingerprint_case(dtype, C, E, spots, 32 * E, "(((a+b)+(c+d))+e)", 2)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_lookback_order(dtype):
    """First elements of chunks 0..3.  Chunk 3's look-back lanes read chunks
    2,1,0: Excl(3) = PT(c, b, a) = (c+b)+a, then d."""
    E, C = scan_geometry(dtype)
    spots = {"a": 0, "b": C, "c": 2 * C, "d": 3 * C}
    _fingerprint_case(dtype, C, E, spots, 3 * C, "(((c+b)+a)+d)", 3)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_anchor(dtype):
    """Chunks 0, 1, 30 in interval 0, its anchor chunk 31, and chunk 32.
    Excl(31): lanes 0 (chunk 30), 29 (chunk 1), 30 (chunk 0) -> c+(b+a);
    A(0) = Excl(31) + d; chunk 32 starts from A(0), then e."""
    E, C = scan_geometry(dtype)
    spots = {"a": 0, "b": C, "c": 30 * C, "d": 31 * C, "e": 32 * C}
    _fingerprint_case(dtype, C, E, spots, 32 * C, "(((c+(b+a))+d)+e)", 4)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_after_anchor(dtype):
    """Chunk 33 (k=1, j=1): lane 0 reads Agg(32), lane 1 the anchor A(0)."""
    E, C = scan_geometry(dtype)
    spots = {"a": 5 * C + 7, "d": 31 * C, "e": 32 * C + 1, "f": 33 * C + 2}
    # A(0) = Excl(31) + d with Excl(31) = a (only chunk 5 is nonzero before it)
    _fingerprint_case(dtype, C, E, spots, 33 * C + 2, "((e+(a+d))+f)", 5)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_element_fold_after_carry(dtype):
    """The element step.  Lane 0 of warp 1 holds b then c, and its carry is
    the warp prefix WX[1] = a.  Each element is the running fold that starts
    from the carry, so the second one is ((a+b)+c), not the carry plus the
    lane's own prefix, (a+(b+c))."""
    E, C = scan_geometry(dtype)
    spots = {"a": 0, "b": 32 * E, "c": 32 * E + 1}
    _fingerprint_case(dtype, C, E, spots, 32 * E + 1, "((a+b)+c)", 6)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_fingerprint_element_fold_full_carry(dtype):
    """Chunk 1, warp 5, lane 3 holds d (element 0) and e (element 2).  Its
    carry is ((Excl(1) + WX[5]) + LX[3]) with Excl(1) = a (chunk 0),
    WX[5] = b (warp 3 of chunk 1) and LX[3] = c (lane 2 of warp 5); d and e
    are then folded in one at a time: ((((a+b)+c)+d)+e), where the
    carry-plus-lane-prefix form would give (((a+b)+c)+(d+e))."""
    E, C = scan_geometry(dtype)
    w5 = C + 5 * 32 * E
    spots = {"a": 7, "b": C + 3 * 32 * E + 1, "c": w5 + 2 * E + 4,
             "d": w5 + 3 * E, "e": w5 + 3 * E + 2}
    _fingerprint_case(dtype, C, E, spots, w5 + 3 * E + 2, "((((a+b)+c)+d)+e)", 7)


def _segmented_fingerprint_case(dtype, E, offsets, outside, spots, query, bracket, seed):
    """Like _fingerprint_case for det_segmented_scan: ``outside`` holds
    positions before the query's segment head, filled with large values that
    must not reach the result."""
    rng = np.random.default_rng(seed)
    order = sorted(spots, key=lambda nm: spots[nm])
    vals = distinguishing_values(order, dtype, rng, canonical(parse(bracket), order))
    n = int(offsets[-1])
    x = np.full(n, -0.0, dtype)
    for p in outside:
        x[p] = dtype(1024.0 + p)
    for nm, p in spots.items():
        x[p] = vals[nm]
    y = oracle.det_segmented_scan(x, np.asarray(offsets, np.int64))
    assert same_bits(y[query], evaluate(parse(bracket), vals, dtype)), (bracket, y[query])
    hits = [t for t in all_trees(order) if same_bits(evaluate(t, vals, dtype), y[query])]
    assert len(hits) == 1


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_fingerprint_element_fold_full_carry(dtype):
    """The segmented element step.  The segment starts at element 3 of chunk
    0 (a); chunk 0's element 1 (before the head) is large and must vanish.
    In chunk 1, b sits in warp 2 and c in lane 1 of warp 4; lane 2 of warp 4
    holds d (element 0) and e (element 3).  The carry is
    ((Excl(1) (+) WX[4]) (+) LX[2]) = ((a+b)+c), and d and e are folded in
    one at a time: ((((a+b)+c)+d)+e)."""
    E, C = scan_geometry(dtype)
    w4 = C + 4 * 32 * E
    spots = {"a": 3, "b": C + 2 * 32 * E + 5, "c": w4 + E + 1,
             "d": w4 + 2 * E, "e": w4 + 2 * E + 3}
    n = w4 + 3 * E + 9
    _segmented_fingerprint_case(dtype, E, [0, 3, n], [1], spots, w4 + 2 * E + 3,
                                "((((a+b)+c)+d)+e)", 8)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_fingerprint_element_fold_in_lane_head(dtype):
    """A head inside a lane: lane 1 of warp 1 holds junk, then the head a,
    then b and c.  The lane's carry (warp 0 and lane 0 of warp 1, all
    before the head) and the junk must vanish at a, and b and c fold in
    one at a time: ((a+b)+c)."""
    E, C = scan_geometry(dtype)
    lane = 32 * E + E
    spots = {"a": lane + 2, "b": lane + 4, "c": lane + 5}
    n = lane + E + 3
    _segmented_fingerprint_case(dtype, E, [0, lane + 2, n], [0, 32 * E + 1, lane],
                                spots, lane + 5, "((a+b)+c)", 9)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_scan_exclusive_is_shifted_inclusive_and_reverse(dtype):
    x = workloads.scan_input(n=100000, dtype=dtype)
    inc, tot = oracle.det_scan(x)
    exc, _ = oracle.det_scan(x, oracle.SCAN_EXCLUSIVE)
    assert same_bits(exc[1:], inc[:-1]) and same_bits(exc[0], dtype(0.0))
    assert same_bits(tot, inc[-1])
    rinc, rtot = oracle.det_scan(x, oracle.SCAN_REVERSE)
    assert same_bits(rinc, oracle.det_scan(x[::-1].copy())[0][::-1])
    assert same_bits(rtot, rinc[0])


@pytest.mark.parametrize("dtype,u", [(F32, 2.0 ** -24), (F64, 2.0 ** -53)])
def test_scan_error_bound_vs_exact_prefix(dtype, u):
    E, C = scan_geometry(dtype)
    n = 2 * 32 * C + 999
    x = workloads.scan_input(n=n, dtype=dtype)
    y, _ = oracle.det_scan(x)
    xd = x.astype(np.float64)
    for i in list(range(0, n, n // 13)) + [n - 1]:
        exact = math.fsum(xd[: i + 1])
        k = (i // C) // 32
        depth = 2 * E + 18 + 6 * (k + 1)      # a-priori depth of the frozen order
        gamma = depth * u / (1 - depth * u)
        assert abs(float(y[i]) - exact) <= gamma * math.fsum(np.abs(xd[: i + 1]))


# --------------------------------------------------------------------------
# det_segmented_scan


@pytest.mark.parametrize("dtype", [F32, F64])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_segscan_one_segment_equals_scan(dtype, flags):
    _, C = scan_geometry(dtype)
    n = 33 * C + 5
    x = workloads.scan_input(n=n, dtype=dtype)
    y = oracle.det_segmented_scan(x, np.array([0, n], np.int64), flags)
    assert same_bits(y, oracle.det_scan(x, flags)[0])


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_singletons(dtype):
    x = workloads.scan_input(n=70000, dtype=dtype)
    off = np.arange(x.size + 1, dtype=np.int64)
    for flags in (0, 2):
        assert same_bits(oracle.det_segmented_scan(x, off, flags), x)
    for flags in (1, 3):
        assert same_bits(oracle.det_segmented_scan(x, off, flags), np.zeros_like(x))


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_ones_closed_form(dtype):
    _, C = scan_geometry(dtype)
    n = 33 * C + 101
    off = workloads.segment_offsets(n, mean=5000, seed=9)
    off = np.unique(np.concatenate([off, [off[3]]]))      # keep sorted
    off = np.insert(off, 5, off[5])                       # an empty segment
    x = np.ones(n, dtype)
    seg = np.searchsorted(off, np.arange(n), side="right") - 1
    start, end = off[seg], off[seg + 1]
    pos = np.arange(n) - start
    assert np.array_equal(oracle.det_segmented_scan(x, off, 0), pos + 1)
    assert np.array_equal(oracle.det_segmented_scan(x, off, 1), pos)
    assert np.array_equal(oracle.det_segmented_scan(x, off, 2), end - np.arange(n))
    assert np.array_equal(oracle.det_segmented_scan(x, off, 3), end - np.arange(n) - 1)


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_is_masked_scan(dtype):
    """Each segment's result equals the full scan of a copy in which every
    element before the segment's head is absent (-0.0)."""
    _, C = scan_geometry(dtype)
    n = 34 * C + 321
    x = workloads.scan_input(n=n, dtype=dtype)
    off = workloads.segment_offsets(n, mean=3 * C, seed=3)
    y = oracle.det_segmented_scan(x, off)
    for s in range(len(off) - 1):
        a, b = int(off[s]), int(off[s + 1])
        if a == b:
            continue
        masked = x.copy()
        masked[:a] = -0.0
        ref, _ = oracle.det_scan(masked[:b].copy())
        assert same_bits(y[a:b], ref[a:b]), s


@pytest.mark.parametrize("dtype", [F32, F64])
def test_segscan_reverse_is_scan_of_reversed_segments(dtype):
    n = 50001
    x = workloads.scan_input(n=n, dtype=dtype)
    off = workloads.fixed_segment_offsets(n, 7777)
    roff = (n - off[::-1]).astype(np.int64)
    for excl in (0, 1):
        y = oracle.det_segmented_scan(x, off, 2 | excl)
        ref = oracle.det_segmented_scan(x[::-1].copy(), roff, excl)[::-1]
        assert same_bits(y, ref)


def test_segscan_rejects_bad_offsets():
    x = np.ones(10, F32)
    with pytest.raises(ValueError):
        oracle.det_segmented_scan(x, np.array([0, 5, 4, 10], np.int64))
    with pytest.raises(ValueError):
        oracle.det_segmented_scan(x, np.array([0, 9], np.int64))
