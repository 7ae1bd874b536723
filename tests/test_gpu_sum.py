"""det_sum on the GPU against the CPU oracle: bit for bit, at every block
size, over repeated runs, on misaligned inputs, and at the full workload size."""
import hashlib
import math

import numpy as np
import pytest

import oracle
from deterministic_floating_point_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DT = {np.float32: torch.float32, np.float64: torch.float64}
BLOCKS = [0, 128, 256, 512, 1024]


@pytest.fixture(scope="module")
def det():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build, det as d
    _build.build()
    return d


def gpu_sum(det, x_np, block_threads=0, offset=0):
    t = torch.from_numpy(x_np).cuda()
    if offset:
        # misaligned view: copy into a buffer at an element offset
        buf = torch.empty(t.numel() + offset, dtype=t.dtype, device="cuda")
        buf[offset:] = t
        t = buf[offset:]
    return det.det_sum(t, block_threads=block_threads).cpu().numpy()[0]


def bits(v, dtype):
    return np.array([v], dtype=dtype).tobytes()


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 31, 32, 33, 511, 512, 1023, 1024, 1025, 4095, 4097,
                               65536 + 17, (1 << 20), (1 << 20) + 7, 3 * (1 << 20) + 13])
def test_sum_matches_oracle(det, n, dtype):
    x = workloads.sum_input(n=n, dtype=dtype, seed=n)
    want = bits(oracle.det_sum(x), dtype)
    for bt in BLOCKS:
        assert bits(gpu_sum(det, x, bt), dtype) == want, bt


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("offset", [1, 3])
def test_sum_misaligned_input(det, dtype, offset):
    x = workloads.sum_input(n=200_001, dtype=dtype, seed=5)
    assert bits(gpu_sum(det, x, 0, offset), dtype) == bits(oracle.det_sum(x), dtype)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_sum_signed_zero_and_fingerprint(det, dtype):
    z = np.full(4097, -0.0, dtype=dtype)
    assert bits(gpu_sum(det, z), dtype) == bits(-0.0, dtype)
    assert bits(gpu_sum(det, np.zeros(0, dtype)), dtype) == bits(0.0, dtype)
    rng = np.random.default_rng(3)
    x = np.full(1 << 20, -0.0, dtype=dtype)
    pos = [2, 3, 4, 1000, 4096, 4097, (1 << 20) - 1]
    x[pos] = (rng.standard_normal(len(pos)) * 2.0 ** rng.integers(-8, 8, len(pos))).astype(dtype)
    assert bits(gpu_sum(det, x), dtype) == bits(oracle.det_sum(x), dtype)


@pytest.mark.parametrize("dtype,bound", [(np.float32, 2e-6), (np.float64, 1e-14)])
def test_sum_workload_100_runs_three_block_sizes(det, dtype, bound):
    """The 2^20-element uniform[0,12) workload: SHA-256 of the result bits is
    the oracle's over 100 runs at block sizes 128, 256 and 1024 and at the
    default launch."""
    x = workloads.sum_input(dtype=dtype)
    want = hashlib.sha256(bits(oracle.det_sum(x), dtype)).hexdigest()
    t = torch.from_numpy(x).cuda()
    out = torch.empty(1, dtype=t.dtype, device="cuda")
    for bt in (0, 128, 256, 1024):
        hashes = set()
        for _ in range(100):
            det.det_sum(t, out, block_threads=bt)
            hashes.add(hashlib.sha256(out.cpu().numpy().tobytes()).hexdigest())
        assert hashes == {want}, bt
    exact = math.fsum(x.astype(np.float64))
    assert abs(float(out.cpu()[0]) - exact) <= bound * math.fsum(np.abs(x.astype(np.float64)))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_sum_full_size_supplement(det, dtype):
    """n = 2^28, the size the kernel's roofline is measured on, at the default
    launch the bench times and two block sizes."""
    x = workloads.sum_input(n=1 << 28, dtype=dtype, seed=0)
    want = bits(oracle.det_sum(x), dtype)
    for bt in (0, 128, 1024):
        assert bits(gpu_sum(det, x, bt), dtype) == want


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1 << 20, (1 << 24) + 5])
def test_sum_workspace_with_leftover_contents(det, dtype, n):
    """The workspace is never cleared: a call must find its tiles' partials
    among whatever the buffer held before -- small integers in every 32-bit
    half (int32 data), all-ones bytes, random bytes, and the partials of
    earlier calls on other data.  Each call equals the oracle."""
    x = workloads.sum_input(n=n, dtype=dtype, seed=11)
    want = bits(oracle.det_sum(x), dtype)
    other = torch.from_numpy(workloads.sum_input(n=n, dtype=dtype, seed=12)).cuda()
    t = torch.from_numpy(x).cuda()
    out = torch.empty(1, dtype=t.dtype, device="cuda")
    code = 0 if dtype == np.float32 else 1
    ws = det.workspace(det.lib().det_sum_workspace_bytes(n, code), t.device)
    words = ws[: (ws.numel() // 8) * 8].view(torch.int32)
    gen = torch.Generator(device="cuda").manual_seed(5)
    fills = [
        lambda: words.copy_(torch.arange(1, words.numel() + 1, dtype=torch.int32, device="cuda") % 4096),
        lambda: ws.fill_(0xFF),
        lambda: ws.copy_(torch.randint(0, 256, (ws.numel(),), dtype=torch.uint8, device="cuda", generator=gen)),
        lambda: det.det_sum(other, workspace=ws),
    ]
    for fill in fills:
        for _ in range(25):
            fill()
            det.det_sum(t, out, workspace=ws)
            assert bits(out.cpu().numpy()[0], dtype) == want
            assert det.read_status(ws) == 0


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1 << 20, (1 << 24) + 5])
def test_sum_captured_in_a_cuda_graph(det, dtype, n):
    """det_sum captured once in a CUDA graph and replayed over changing inputs
    in the same buffer: every replay equals the oracle on its own input (no
    replay may take another replay's tile partials)."""
    xs = [workloads.sum_input(n=n, dtype=dtype, seed=s) for s in (21, 22, 23)]
    wants = [bits(oracle.det_sum(x), dtype) for x in xs]
    hosts = [torch.from_numpy(x) for x in xs]
    t = torch.empty(n, dtype=DT[dtype], device="cuda")
    out = torch.empty(1, dtype=t.dtype, device="cuda")
    code = 0 if dtype == np.float32 else 1
    ws = det.workspace(det.lib().det_sum_workspace_bytes(n, code), t.device)
    t.copy_(hosts[0])
    det.det_sum(t, out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        det.det_sum(t, out, workspace=ws)
    for r in range(30):
        k = r % 3
        t.copy_(hosts[k])
        g.replay()
        assert bits(out.cpu().numpy()[0], dtype) == wants[k], r
    # the same workspace outside the graph afterwards
    t.copy_(hosts[1])
    det.det_sum(t, out, workspace=ws)
    assert bits(out.cpu().numpy()[0], dtype) == wants[1]
