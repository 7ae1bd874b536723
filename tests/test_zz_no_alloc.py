"""det_sum_noalloc through the C ABI: the sum for callers that cannot
allocate device memory (a plugin inside a runtime that owns all device memory
and offers no allocator, or a loop that must not call cudaMalloc after
start-up).  Its scratch is a static device array inside libdet.so, so the
test checks that two calls in a row -- which share and reuse that array --
each return exactly the bits of det_sum, the entry point that takes a
caller-provided workspace.

This file is named to be collected last, so a stop-at-first-failure run has
already run every other test when it gets here."""
import ctypes

import numpy as np
import pytest

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


def noalloc_sum(det, x, out, stream):
    code = 0 if x.dtype == torch.float32 else 1
    rc = det.lib().det_sum_noalloc(ctypes.c_void_p(x.data_ptr()), x.numel(), code,
                                   ctypes.c_void_p(out.data_ptr()), 0, ctypes.c_void_p(stream))
    assert rc == 0, det.status_string(rc)
    return out


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_noalloc_matches_det_sum_on_two_calls_in_a_row(det, dtype):
    stream = torch.cuda.current_stream().cuda_stream
    # two different sizes so that the second call reuses scratch the first one filled
    for n, seed in ((3_000_017, 1), (1 << 20, 2)):
        x = torch.from_numpy(workloads.sum_input(n=n, dtype=dtype, seed=seed)).cuda()
        out = torch.empty(1, dtype=x.dtype, device="cuda")
        noalloc_sum(det, x, out, stream)
        ref = det.det_sum(x)              # the existing entry point, own workspace
        torch.cuda.synchronize()
        assert out.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes(), n


def test_noalloc_rejects_inputs_beyond_its_limit(det):
    # checked on the host before anything is enqueued, so no memory is touched
    fake = ctypes.c_void_p(1 << 20)
    too_big = (1 << 34) + (1 << 30)
    assert det.lib().det_sum_noalloc(fake, too_big, 0, fake, 0, None) == 3
