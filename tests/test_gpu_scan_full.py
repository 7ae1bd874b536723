"""The persistent scan kernels at sizes where every CTA takes several chunks,
and the segmented scans at the benchmark's size, bit for bit against the CPU
oracle.

The 1,024-thread kernel runs one CTA per SM (plus the anchor-chain CTA) and
hands chunks out round-robin, so only inputs of more than twice that many
chunks make every CTA carry a chunk from one iteration into the next (the
register hand-off, the prefetched stage and head bits, the deferred first
element of exclusive chunks).  The restart kernel is persistent too: more
segments than resident CTAs make each CTA take several."""
import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FLAGS = [0, 1, 2, 3]


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _many_chunks(dtype):
    """An element count of more than 2.5 chunks per worker CTA, ragged tail."""
    C = oracle.scan_chunk_elems(dtype)
    nch = max(420, int(2.7 * (_sms() + 1)))
    n = nch * C + 77
    assert (n // C) >= 2 * (_sms() + 1)
    return n


def _same(got, want, what):
    assert got.tobytes() == want.tobytes(), what


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", FLAGS)
def test_scan_many_chunks_per_cta(det, dtype, flags):
    n = _many_chunks(dtype)
    x_np = workloads.scan_input(n=n, dtype=dtype, seed=40 + flags)
    want, wtot = oracle.det_scan(x_np, flags)
    x = torch.from_numpy(x_np).cuda()
    for bt in (0, 1024, 256):
        y = torch.empty_like(x)
        tot = torch.empty(1, dtype=x.dtype, device="cuda")
        det.det_scan(x, y, flags=flags, total_out=tot, block_threads=bt)
        _same(y.cpu().numpy(), want, (flags, bt))
        _same(tot.cpu().numpy(), np.array([wtot], dtype), (flags, bt, "total"))
    xi = x.clone()
    det.det_scan(xi, xi, flags=flags)                      # in place
    _same(xi.cpu().numpy(), want, (flags, "in place"))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", FLAGS)
def test_segscan_many_chunks_per_cta(det, dtype, flags):
    n = _many_chunks(dtype)
    C = oracle.scan_chunk_elems(dtype)
    x_np = workloads.scan_input(n=n, dtype=dtype, seed=50 + flags)
    off_np = workloads.segment_offsets(n, mean=4096, seed=50)
    # an empty segment, a segment of one element and one of several anchor intervals
    cut = int(off_np[100])
    off_np = np.unique(np.concatenate([off_np, [cut, cut + 1, cut + 1 + 70 * C]]))
    off_np = np.insert(off_np, 7, off_np[7]).astype(np.int64)
    want = oracle.det_segmented_scan(x_np, off_np, flags)
    x = torch.from_numpy(x_np).cuda()
    off = torch.from_numpy(off_np).cuda()
    for bt in (0, 256):
        y = det.det_segmented_scan(x, off, flags=flags, block_threads=bt)
        _same(y.cpu().numpy(), want, (flags, bt))
    xi = x.clone()
    det.det_segmented_scan(xi, off, xi, flags=flags)       # in place
    _same(xi.cpu().numpy(), want, (flags, "in place"))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", [0, 3])
def test_segscan_full_size(det, dtype, flags):
    """The benchmark's segmented workload: 2^28 lognormal values, geometric
    segments of mean 4,096."""
    x_np = workloads.scan_input(n=workloads.SCAN_N, dtype=dtype)
    off_np = workloads.segment_offsets(x_np.size)
    want = oracle.det_segmented_scan(x_np, off_np, flags)
    got = det.det_segmented_scan(torch.from_numpy(x_np).cuda(), torch.from_numpy(off_np).cuda(), flags=flags)
    _same(got.cpu().numpy(), want, flags)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("flags", FLAGS)
def test_restart_more_segments_than_ctas(det, dtype, flags):
    """Per-segment restart with about 8,000 segments -- more than the
    resident CTAs of the persistent restart kernel at any occupancy (at most
    2,048 threads per SM) -- plus segments that span anchor intervals."""
    C = oracle.scan_chunk_elems(dtype)
    rng = np.random.default_rng(60 + flags)
    lens = list(rng.geometric(1 / 4096, 8000)) + [33 * C + 9, 0, 1, C]
    rng.shuffle(lens)
    off_np = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    assert off_np.size - 1 > 2048 // 128 * _sms()
    x_np = rng.lognormal(0, 1, int(off_np[-1])).astype(dtype)
    want = oracle.det_segmented_scan(x_np, off_np, flags | oracle.SCAN_SEGMENT_RESTART)
    got = det.det_segmented_scan(torch.from_numpy(x_np).cuda(), torch.from_numpy(off_np).cuda(),
                                 flags=flags | det.SCAN_SEGMENT_RESTART)
    _same(got.cpu().numpy(), want, flags)
