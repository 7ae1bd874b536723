"""det_scan / det_segmented_scan on the GPU against the CPU oracle, bit for
bit: every flag combination, every block size, ragged sizes across lanes,
warps, chunks and anchor intervals, in place, segmented with empty and
one-element segments, repeated runs, and the full workload size."""
import hashlib

import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FLAGS = [0, 1, 2, 3]
BLOCKS = [0, 128, 256, 512, 1024]


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def chunk(dtype):
    return oracle.scan_chunk_elems(dtype)


def run_scan(det, x_np, flags, bt=0, inplace=False, with_total=False):
    x = torch.from_numpy(x_np).cuda()
    y = x if inplace else torch.empty_like(x)
    tot = torch.empty(1, dtype=x.dtype, device="cuda") if with_total else None
    ws = det.workspace(det.lib().det_scan_workspace_bytes(x.numel(), 0 if x.dtype == torch.float32 else 1),
                       x.device)
    det.det_scan(x, y, flags=flags, total_out=tot, block_threads=bt, workspace=ws)
    assert det.read_status(ws) == 0
    return y.cpu().numpy(), (tot.cpu().numpy()[0] if with_total else None)


def run_segscan(det, x_np, off_np, flags, bt=0, inplace=False):
    x = torch.from_numpy(x_np).cuda()
    off = torch.from_numpy(off_np).cuda()
    y = x if inplace else torch.empty_like(x)
    ws = det.workspace(det.lib().det_segmented_scan_workspace_bytes(
        x.numel(), off.numel() - 1, 0 if x.dtype == torch.float32 else 1), x.device)
    det.det_segmented_scan(x, off, y, flags=flags, block_threads=bt, workspace=ws)
    assert det.read_status(ws) == 0
    return y.cpu().numpy()


def sizes(dtype):
    C = chunk(dtype)
    E = oracle.scan_lane_elems(dtype)
    return [1, 2, E - 1, E + 1, 32 * E + 3, C - 1, C, C + 1, 3 * C + 5, 32 * C, 33 * C + 7, 65 * C + 13]


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", FLAGS)
def test_scan_matches_oracle(det, dtype, flags):
    for n in sizes(dtype):
        x = workloads.scan_input(n=n, dtype=dtype, seed=n % 1000)
        want, wtot = oracle.det_scan(x, flags)
        for bt in (0, 256):
            got, tot = run_scan(det, x, flags, bt, with_total=True)
            assert got.tobytes() == want.tobytes(), (n, bt)
            assert np.array([tot]).tobytes() == np.array([wtot]).tobytes(), (n, bt)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bt", BLOCKS)
def test_scan_block_sizes_and_in_place(det, dtype, bt):
    C = chunk(dtype)
    n = 34 * C + 321
    x = workloads.scan_input(n=n, dtype=dtype, seed=7)
    for flags in FLAGS:
        want, _ = oracle.det_scan(x, flags)
        got, _ = run_scan(det, x, flags, bt, inplace=True)
        assert got.tobytes() == want.tobytes(), flags


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_scan_small_workload_100_runs(det, dtype):
    """The 164,738-element lognormal input: 100 runs at three block sizes and
    the default launch (for f64 the one-cluster path) give the oracle's
    SHA-256 for every flag combination."""
    x_np = workloads.scan_input(dtype=dtype)
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty_like(x)
    ws = det.workspace(det.lib().det_scan_workspace_bytes(x.numel(), 0 if dtype == np.float32 else 1), x.device)
    for flags in FLAGS:
        want = hashlib.sha256(oracle.det_scan(x_np, flags)[0].tobytes()).hexdigest()
        for bt in (0, 128, 256, 1024):
            seen = set()
            for _ in range(100):
                det.det_scan(x, y, flags=flags, block_threads=bt, workspace=ws)
                seen.add(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
            assert seen == {want}, (flags, bt)
    assert det.read_status(ws) == 0


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", FLAGS)
def test_segscan_matches_oracle(det, dtype, flags):
    C = chunk(dtype)
    for n, off in [
        (33 * C + 7, workloads.segment_offsets(33 * C + 7, mean=4096, seed=1)),
        (200_000, workloads.fixed_segment_offsets(200_000, 65_537)),
        (5 * C + 3, np.array([0, 0, 1, 1, 2, C - 1, C, C, 3 * C + 1, 5 * C + 3, 5 * C + 3], np.int64)),
        (3 * C, np.array([0, 3 * C], np.int64)),
        (70_001, np.arange(70_002, dtype=np.int64)),
    ]:
        x = workloads.scan_input(n=n, dtype=dtype, seed=3)
        want = oracle.det_segmented_scan(x, off, flags)
        for bt in (0, 128):
            got = run_segscan(det, x, off, flags, bt)
            assert got.tobytes() == want.tobytes(), (n, bt)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_segscan_in_place_and_block_sizes(det, dtype):
    C = chunk(dtype)
    n = 40 * C + 99
    x = workloads.scan_input(n=n, dtype=dtype, seed=11)
    off = workloads.segment_offsets(n, mean=4096, seed=2)
    for flags in FLAGS:
        want = oracle.det_segmented_scan(x, off, flags)
        for bt in (256, 512, 1024):
            got = run_segscan(det, x, off, flags, bt, inplace=True)
            assert got.tobytes() == want.tobytes(), (flags, bt)


def test_scan_zero_length(det):
    x = torch.empty(0, dtype=torch.float32, device="cuda")
    tot = torch.full((1,), 7.0, device="cuda")
    det.det_scan(x, torch.empty_like(x), total_out=tot)
    assert tot.item() == 0.0


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_scan_full_size(det, dtype):
    """n = 2^28 lognormal: the benchmark's size, forward inclusive and
    reverse exclusive, bit for bit against the oracle."""
    n = 1 << 28
    x = workloads.scan_input(n=n, dtype=dtype, seed=4)
    for flags in (0, 3):
        want, _ = oracle.det_scan(x, flags)
        got, _ = run_scan(det, x, flags)
        assert got.tobytes() == want.tobytes(), flags
        del want, got
