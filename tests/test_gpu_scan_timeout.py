"""The bounded look-back waits of det_scan / det_segmented_scan, made to run
out on purpose: a test hook withholds one chunk's aggregate, so the chunks
that read it (and the anchor chain) wait until a short limit expires.  The
launch must end by itself, the status word must say
DET_ERR_LOOKBACK_TIMEOUT, and the next call must be correct again.  Nothing
here faults or hangs the GPU: every wait is bounded in time, and the
withheld value is simply never written."""
import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOOKBACK_TIMEOUT = 5    # DET_ERR_LOOKBACK_TIMEOUT
LIMIT_NS = 5_000_000    # 5 ms


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def _ws(det, x, nseg=None):
    code = 0 if x.dtype == torch.float32 else 1
    nbytes = (det.lib().det_scan_workspace_bytes(x.numel(), code) if nseg is None
              else det.lib().det_segmented_scan_workspace_bytes(x.numel(), nseg, code))
    return det.workspace(nbytes, x.device)


def _call(det, x, y, off, flags, bt, ws):
    if off is None:
        det.det_scan(x, y, flags=flags, block_threads=bt, workspace=ws)
    else:
        det.det_segmented_scan(x, off, y, flags=flags, block_threads=bt, workspace=ws)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bt", [0, 256])
@pytest.mark.parametrize("segmented", [False, True])
@pytest.mark.parametrize("flags", [0, 3])
def test_lookback_wait_runs_out_and_is_reported(det, dtype, bt, segmented, flags):
    C = oracle.scan_chunk_elems(dtype)
    n = 80 * C + 5                       # three anchor intervals
    x_np = workloads.scan_input(n=n, dtype=dtype, seed=21)
    off_np = workloads.segment_offsets(n, mean=4096, seed=21) if segmented else None
    x = torch.from_numpy(x_np).cuda()
    off = torch.from_numpy(off_np).cuda() if segmented else None
    y = torch.empty_like(x)
    nseg = None if off_np is None else off_np.size - 1
    lib = det.lib()
    ws = _ws(det, x, nseg)
    assert lib.det_test_scan_withhold(37, LIMIT_NS) == 0   # chunk 37: interval 1, read by 38..68 and the chain
    try:
        _call(det, x, y, off, flags, bt, ws)
        assert det.read_status(ws) == LOOKBACK_TIMEOUT
    finally:
        assert lib.det_test_scan_withhold(-1, 0) == 0
    # the context is still usable: the next calls (same and fresh workspace) are exact
    want = (oracle.det_scan(x_np, flags)[0] if off_np is None
            else oracle.det_segmented_scan(x_np, off_np, flags))
    for w in (ws, _ws(det, x, nseg)):
        _call(det, x, y, off, flags, bt, w)
        assert det.read_status(w) == 0
        assert y.cpu().numpy().tobytes() == want.tobytes()


def test_withheld_chunk_past_the_end_changes_nothing(det):
    """A hook aimed past the last chunk withholds nothing: no wait runs out."""
    x_np = workloads.scan_input(n=3 * oracle.scan_chunk_elems(np.float32) + 1, dtype=np.float32)
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty_like(x)
    ws = _ws(det, x)
    lib = det.lib()
    assert lib.det_test_scan_withhold(1000, LIMIT_NS) == 0
    try:
        det.det_scan(x, y, workspace=ws)
        assert det.read_status(ws) == 0
    finally:
        lib.det_test_scan_withhold(-1, 0)
    assert y.cpu().numpy().tobytes() == oracle.det_scan(x_np)[0].tobytes()
