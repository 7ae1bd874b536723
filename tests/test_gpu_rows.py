"""det_scatter_add_rows on the GPU against the CPU oracle: destination rows and
previous rows bit for bit, the page's worked example, skipped rows, offsets,
odd row lengths, block sizes, repeated runs and the full workload size."""
import hashlib
import json
import os

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


def gpu_rows(det, dst0, idx, src, off=0, bt=0, with_prev=True):
    dst = torch.from_numpy(np.array(dst0, copy=True)).cuda()
    s = torch.from_numpy(src).cuda()
    i = torch.from_numpy(idx).cuda()
    prev = torch.full_like(s, 99.0) if with_prev else None
    ws = det.workspace(det.lib().det_scatter_add_rows_workspace_bytes(
        src.shape[0], dst0.shape[0], dst0.shape[1], 0 if src.dtype == np.float32 else 1), s.device)
    det.det_scatter_add_rows(dst, i, s, row_offset=off, prev_out=prev, block_threads=bt, workspace=ws)
    assert det.read_status(ws) == 0
    return dst.cpu().numpy(), (prev.cpu().numpy() if with_prev else None)


def check(det, dst0, idx, src, off=0, bts=(0,)):
    want_dst, want_prev = oracle.det_scatter_add_rows(dst0, idx, src, row_offset=off)
    for bt in bts:
        dst, prev = gpu_rows(det, dst0, idx, src, off, bt)
        assert dst.tobytes() == want_dst.tobytes(), bt
        assert prev.tobytes() == want_prev.tobytes(), bt


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_tile_example_golden(det, dtype, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tile_atomic_add_indexed_example.json")))
    dst, prev = gpu_rows(det, np.array(g["y"], dtype), np.array(g["indices"], np.int32), np.array(g["x"], dtype))
    assert dst.tolist() == g["expected_y"]
    assert prev.tolist() == g["expected_previous"]


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("M,R,W,off", [(1, 1, 1, 0), (100, 7, 3, 0), (5000, 64, 64, 0), (20_000, 300, 65, 2),
                                       (40_000, 1000, 130, -5), (3000, 4, 1, 0), (70_000, 65_536, 64, 0),
                                       (9000, 3, 200, 1)])
def test_rows_match_oracle(det, dtype, M, R, W, off):
    rng = np.random.default_rng(M + W)
    src = rng.standard_normal((M, W)).astype(dtype)
    idx = rng.integers(-3, R + 3, M, dtype=np.int32)
    dst0 = rng.standard_normal((R, W)).astype(dtype)
    check(det, dst0, idx, src, off)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("bt", [0, 128, 256, 512, 1024])
def test_rows_block_sizes_and_long_groups(det, dtype, bt):
    rng = np.random.default_rng(3)
    M, R, W = 50_000, 5, 64          # about 10,000 source rows per destination
    src = rng.standard_normal((M, W)).astype(dtype)
    idx = rng.integers(0, R, M, dtype=np.int32)
    dst0 = rng.standard_normal((R, W)).astype(dtype)
    check(det, dst0, idx, src, bts=(bt,))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_rows_without_prev_and_empty(det, dtype):
    rng = np.random.default_rng(5)
    src = rng.standard_normal((1000, 8)).astype(dtype)
    idx = rng.integers(0, 10, 1000, dtype=np.int32)
    dst0 = rng.standard_normal((10, 8)).astype(dtype)
    want, _ = oracle.det_scatter_add_rows(dst0, idx, src)
    dst, _ = gpu_rows(det, dst0, idx, src, with_prev=False)
    assert dst.tobytes() == want.tobytes()
    dst, prev = gpu_rows(det, dst0, np.full(1000, 50, np.int32), src)   # every row skipped
    assert dst.tobytes() == dst0.tobytes() and not prev.any()


def test_rows_workload_full_size_100_runs(det):
    """src 2^20 x 64 f32 N(0,1), rows uniform over a 65,536 x 64 destination:
    at each of the block sizes 128, 256, 1024 and the default, 100 runs; the
    first one's destination and previous rows hash to the oracle's (SHA-256),
    and every later run's bits equal the first's (compared on the device)."""
    src, idx, dst0 = workloads.rows_input()
    want_dst, want_prev = oracle.det_scatter_add_rows(dst0, idx, src)
    want = hashlib.sha256(want_dst.tobytes() + want_prev.tobytes()).hexdigest()
    s = torch.from_numpy(src).cuda()
    i = torch.from_numpy(idx).cuda()
    prev = torch.empty_like(s)
    ws = det.workspace(det.lib().det_scatter_add_rows_workspace_bytes(src.shape[0], dst0.shape[0], 64, 0), s.device)
    dst0_d = torch.from_numpy(dst0).cuda()
    for bt in (128, 256, 1024, 0):
        first = None
        for r in range(100):
            dst = dst0_d.clone()
            det.det_scatter_add_rows(dst, i, s, prev_out=prev, block_threads=bt, workspace=ws)
            if first is None:
                got = hashlib.sha256(dst.cpu().numpy().tobytes() + prev.cpu().numpy().tobytes()).hexdigest()
                assert got == want, bt
                first = (dst.view(torch.int32).clone(), prev.view(torch.int32).clone())
            else:
                assert torch.equal(dst.view(torch.int32), first[0]) and \
                    torch.equal(prev.view(torch.int32), first[1]), (bt, r)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("W", [2, 4, 8, 100, 128])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (2, 0), (0, 1)])
@pytest.mark.parametrize("ordered", [False, True])
def test_rows_layouts(det, dtype, W, src_off, dst_off, ordered):
    """Row lengths and base offsets that select each access form: pair
    accesses (even W, every array on a pair boundary) and single columns (an
    odd element offset of dst), each with one long group and many short
    ones."""
    rng = np.random.default_rng(W * 7 + src_off * 3 + dst_off)
    M, R = 30_001, 900
    src = rng.standard_normal((M, W)).astype(dtype)
    idx = rng.integers(-2, R + 2, M, dtype=np.int32)
    idx[:2500] = 11                                        # one long group: many rounds
    dst0 = rng.standard_normal((R, W)).astype(dtype)
    f = oracle.det_scatter_add_rows_ordered if ordered else oracle.det_scatter_add_rows
    want_dst, want_prev = f(dst0, idx, src)
    sbuf = torch.zeros(src_off + M * W, dtype=torch.float32 if dtype == np.float32 else torch.float64, device="cuda")
    dbuf = torch.zeros(dst_off + R * W, dtype=sbuf.dtype, device="cuda")
    s = sbuf[src_off:].view(M, W)
    s.copy_(torch.from_numpy(src))
    dst = dbuf[dst_off:].view(R, W)
    dst.copy_(torch.from_numpy(dst0))
    prev = torch.full_like(s, 99.0)
    ws = det.workspace(det.lib().det_scatter_add_rows_workspace_bytes(M, R, W, 0 if dtype == np.float32 else 1),
                       s.device)
    det.det_scatter_add_rows(dst, torch.from_numpy(idx).cuda(), s, prev_out=prev, workspace=ws, ordered=ordered)
    assert det.read_status(ws) == 0
    assert dst.cpu().numpy().tobytes() == want_dst.tobytes()
    assert prev.cpu().numpy().tobytes() == want_prev.tobytes()
