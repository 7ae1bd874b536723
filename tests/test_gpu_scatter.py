"""det_scatter_add on the GPU against the CPU oracle: output bits, the sort
permutation and the segment offsets all exact, for one- and two-pass key
sizes, skew, out-of-range indices, every block size, repeated runs and the
full workload sizes."""
import hashlib
import json
import os

import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BLOCKS = [0, 128, 256, 512, 1024]


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def gpu_scatter(det, out0, bins, values, bt=0, want_perm=True):
    out = torch.from_numpy(np.array(out0, copy=True)).cuda()
    b = torch.from_numpy(bins).cuda()
    v = torch.from_numpy(values).cuda()
    m = out.numel()
    perm = torch.full((max(1, bins.size),), -7, dtype=torch.int32, device="cuda") if want_perm else None
    seg = torch.empty(m + 1, dtype=torch.int32, device="cuda")
    ws = det.workspace(det.lib().det_scatter_add_workspace_bytes(bins.size, m, 0 if values.dtype == np.float32 else 1),
                       v.device)
    det.det_scatter_add(out, b, v, perm_out=perm, seg_offsets_out=seg, block_threads=bt, workspace=ws)
    assert det.read_status(ws) == 0
    nvalid = int(seg[-1].item())
    return out.cpu().numpy(), (perm[:nvalid].cpu().numpy() if want_perm else None), seg.cpu().numpy()


def check(det, out0, bins, values, bts=(0,)):
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    for bt in bts:
        out, perm, seg = gpu_scatter(det, out0, bins, values, bt)
        assert out.tobytes() == want_out.tobytes(), ("out", bt)
        assert np.array_equal(perm, want_perm), ("perm", bt)
        assert np.array_equal(seg, want_seg), ("seg", bt)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_quickstart_golden(det, dtype, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "quickstart_ones.json")))
    values = np.full(g["n"], g["value"], dtype=dtype)
    bins = np.full(g["n"], g["bin"], dtype=np.int32)
    out, _, _ = gpu_scatter(det, np.zeros(g["out_len"], dtype), bins, values)
    assert out.tolist() == g["expected_out"]


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n,m", [(1, 1), (5, 3), (100, 1024), (5000, 1024), (70_001, 1024), (1_048_583, 1024),
                                 (300_000, 7), (200_000, 65_536), (400_000, 1 << 20), (50_000, 1 << 21),
                                 (10, 1)])
def test_uniform_matches_oracle(det, dtype, n, m):
    values, bins, out0 = workloads.scatter_input(n=n, num_bins=m, dtype=dtype, seed=n % 97)
    out0 = workloads.sum_input(n=m, dtype=dtype, seed=1) - dtype(6.0)
    check(det, out0, bins, values)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_all_in_one_bin_long_segment(det, dtype):
    values, bins, out0 = workloads.scatter_input(n=(1 << 20) + 3, num_bins=8, dtype=dtype, all_in_bin0=True)
    check(det, out0, bins, values, bts=(0, 1024))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_skewed_with_out_of_range(det, dtype):
    values, bins, out0 = workloads.skewed_scatter_input(n=1 << 21, num_bins=1 << 20, dtype=dtype, seed=7)
    check(det, out0, bins, values, bts=(0, 256))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bt", BLOCKS)
def test_block_sizes(det, dtype, bt):
    values, bins, out0 = workloads.skewed_scatter_input(n=300_007, num_bins=5000, dtype=dtype, seed=3)
    check(det, out0, bins, values, bts=(bt,))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_edge_cases(det, dtype):
    # nothing valid, untouched bits (including -0.0) survive
    bins = np.array([-1, 9, -2147483648, 2147483647], dtype=np.int32)
    values = np.array([1, 2, 3, 4], dtype=dtype)
    out0 = np.array([-0.0, 1.5, -0.0], dtype=dtype)
    check(det, out0, bins, values)
    # zero records, zero destinations
    check(det, out0, np.zeros(0, np.int32), np.zeros(0, dtype))
    out, _, seg = gpu_scatter(det, np.zeros(0, dtype), np.array([0, 1], np.int32), np.array([1, 2], dtype))
    assert seg.tolist() == [0]


def test_argument_errors(det):
    v = torch.ones(4, device="cuda")
    b = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, device="cuda")
    with pytest.raises(Exception):
        det.det_scatter_add(out, b, v, block_threads=96)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("variant", ["uniform", "bin0"])
def test_scatter_workload_100_runs(det, dtype, variant):
    """n = 2^24 N(0,1) into 1,024 uniform bins (and all in bin 0): at each of
    the block sizes 128, 256, 1024 and the default, 100 runs; the first one's
    output, permutation and offsets hash to the oracle's (SHA-256), and every
    later run's bits equal the first's (compared on the device)."""
    values, bins, out0 = workloads.scatter_input(dtype=dtype, all_in_bin0=(variant == "bin0"))
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    want = hashlib.sha256(want_out.tobytes() + want_perm.tobytes() + want_seg.tobytes()).hexdigest()
    v = torch.from_numpy(values).cuda()
    b = torch.from_numpy(bins).cuda()
    m = out0.size
    perm = torch.empty(bins.size, dtype=torch.int32, device="cuda")
    seg = torch.empty(m + 1, dtype=torch.int32, device="cuda")
    ws = det.workspace(det.lib().det_scatter_add_workspace_bytes(bins.size, m, 0 if dtype == np.float32 else 1),
                       v.device)
    out0_d = torch.from_numpy(out0).cuda()
    ibits = torch.int32 if dtype == np.float32 else torch.int64
    for bt in (128, 256, 1024, 0):
        first = None
        for r in range(100):
            out = out0_d.clone()
            det.det_scatter_add(out, b, v, perm_out=perm, seg_offsets_out=seg, block_threads=bt, workspace=ws)
            if first is None:
                blob = out.cpu().numpy().tobytes() + perm.cpu().numpy().tobytes() + seg.cpu().numpy().tobytes()
                assert hashlib.sha256(blob).hexdigest() == want, bt
                first = (out.view(ibits).clone(), perm.clone(), seg.clone())
            else:
                assert torch.equal(out.view(ibits), first[0]) and torch.equal(perm, first[1]) \
                    and torch.equal(seg, first[2]), (bt, r)
    assert det.read_status(ws) == 0


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_skewed_workload_full_size(det, dtype):
    """n = 2^26 N(0,1), Zipf(1.1) over 2^20 bins, 5 % out of range."""
    values, bins, out0 = workloads.skewed_scatter_input(dtype=dtype)
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    out, perm, seg = gpu_scatter(det, out0, bins, values, 0)
    assert out.tobytes() == want_out.tobytes()
    assert np.array_equal(seg, want_seg)
    assert np.array_equal(perm, want_perm)


@pytest.mark.parametrize("n,m", [((1 << 25) + 1357, 1024), ((1 << 25) + 1357, 1 << 20), ((1 << 26) + 999, 1024)])
def test_many_tiles(det, n, m):
    """Sorts of many tiles: with 4,096-record tiles (block_threads 128),
    2^25 + 1,357 records make 8,193 tiles and 2^26 + 999 records 16,385, so
    the column scan reads each tile group in several batches and the last
    tile is ragged; one- and two-pass keys."""
    values, bins, out0 = workloads.scatter_input(n=n, num_bins=m, dtype=np.float32, seed=n % 89)
    check(det, out0, bins, values, bts=(128,))
