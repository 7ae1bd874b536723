"""det_scatter_add against the CPU oracle over destination ranges and input
sizes: one-pass digit sorts of every width up to 10 bits and two-pass sorts
above, ragged last tiles of both tile sizes, dropped records, runs of equal
destinations, with and without the permutation."""
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


def run(det, out0, bins, values, bt, want_perm):
    out = torch.from_numpy(np.array(out0, copy=True)).cuda()
    b = torch.from_numpy(bins).cuda()
    v = torch.from_numpy(values).cuda()
    m = out.numel()
    perm = torch.full((max(1, bins.size),), -7, dtype=torch.int32, device="cuda") if want_perm else None
    seg = torch.empty(m + 1, dtype=torch.int32, device="cuda")
    code = 0 if values.dtype == np.float32 else 1
    ws = det.workspace(det.lib().det_scatter_add_workspace_bytes(bins.size, m, code), v.device)
    det.det_scatter_add(out, b, v, perm_out=perm, seg_offsets_out=seg, block_threads=bt, workspace=ws)
    assert det.read_status(ws) == 0
    nvalid = int(seg[-1].item())
    return out.cpu().numpy(), (perm[:nvalid].cpu().numpy() if want_perm else None), seg.cpu().numpy()


def mixed_bins(rng, n, m):
    """Uniform destinations with 3 % dropped (negative or past the end) and
    runs of a repeated destination."""
    bins = rng.integers(0, m, n, dtype=np.int64)
    drop = rng.random(n) < 0.03
    bins[drop] = np.where(rng.random(int(drop.sum())) < 0.5, -1 - rng.integers(0, 5, int(drop.sum())),
                          m + rng.integers(0, 5, int(drop.sum())))
    starts = rng.integers(0, max(1, n - 600), 8)
    for s in starts:
        bins[s:s + 500] = rng.integers(0, m)
    return bins.astype(np.int32)


# m covers one-pass digits of 0 to 10 bits and two-pass sorts of 11 and 12 bits
@pytest.mark.parametrize("m", [1, 2, 16, 17, 32, 33, 64, 65, 256, 257, 1024, 1025, 4096])
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_digit_widths(det, m, dtype):
    rng = np.random.default_rng(m)
    n = 3 * 4096 + 77
    bins = mixed_bins(rng, n, m)
    values = workloads.sum_input(n=n, dtype=dtype, seed=m + 11)
    out0 = workloads.sum_input(n=m, dtype=dtype, seed=2) - dtype(3.0)
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    for bt in (0, 128, 256):
        for want in (False, True):
            out, perm, seg = run(det, out0, bins, values, bt, want)
            assert out.tobytes() == want_out.tobytes(), (bt, want)
            assert np.array_equal(seg, want_seg), (bt, want)
            if want:
                assert np.array_equal(perm, want_perm), bt


@pytest.mark.parametrize("n", [1, 15, 16, 17, 2047, 2048, 2049, 4095, 4096, 4097, 1 << 20, (1 << 22) + 5])
def test_ragged_sizes(det, n):
    rng = np.random.default_rng(n % 1000)
    m = 1000
    bins = mixed_bins(rng, n, m) if n > 600 else rng.integers(-2, m + 2, n).astype(np.int32)
    values = workloads.sum_input(n=n, dtype=np.float32, seed=5)
    out0 = np.zeros(m, np.float32)
    want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
    for bt in (0, 256):
        out, perm, seg = run(det, out0, bins, values, bt, True)
        assert out.tobytes() == want_out.tobytes(), bt
        assert np.array_equal(seg, want_seg), bt
        assert np.array_equal(perm, want_perm), bt


def test_all_dropped_and_all_one_key(det):
    n = 50_000
    values = workloads.sum_input(n=n, dtype=np.float32, seed=9)
    out0 = np.full(700, -0.0, np.float32)
    for bins in (np.full(n, -1, np.int32), np.full(n, 700, np.int32), np.full(n, 699, np.int32),
                 np.zeros(n, np.int32)):
        want_out, want_perm, want_seg = oracle.det_scatter_add(out0, bins, values)
        out, perm, seg = run(det, out0, bins, values, 0, True)
        assert out.tobytes() == want_out.tobytes()
        assert np.array_equal(seg, want_seg)
        assert np.array_equal(perm, want_perm)
