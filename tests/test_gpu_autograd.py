"""det_gather_rows and the autograd gather: forward equal to the oracle's
gather, gradient bit-identical to the oracle's scatter-add of the output
gradient (the pages' backward example), on every run and launch shape."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ag():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_floating_point_gb300 import _build
    _build.build()
    from deterministic_floating_point_gb300 import autograd, det
    return autograd, det


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("W", [1, 3, 64, 100])
def test_gather_rows_forward(ag, dtype, W):
    _, det = ag
    rng = np.random.default_rng(60 + W)
    src = rng.standard_normal((5000, W) if W > 1 else 5000).astype(dtype)
    idx = rng.integers(-7, 5007, 100_003).astype(np.int32)
    want = oracle.det_gather_rows(src, idx)
    for bt in (128, 256, 1024):
        got = det.det_gather_rows(torch.from_numpy(src).cuda(), torch.from_numpy(idx).cuda(), block_threads=bt)
        assert np.array_equal(_bits(got.cpu().numpy()), _bits(want))
    got = det.det_gather_rows(torch.from_numpy(src).cuda(), torch.from_numpy(idx + 2).cuda(), row_offset=-2)
    assert np.array_equal(_bits(got.cpu().numpy()), _bits(want))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("W", [1, 64])
@pytest.mark.parametrize("row_offset", [0, 5])
def test_gather_backward_is_the_deterministic_scatter(ag, dtype, W, row_offset):
    autograd, _ = ag
    rng = np.random.default_rng(70 + W + row_offset)
    n_src, n = 3000, 200_000
    src = rng.standard_normal((n_src, W) if W > 1 else n_src).astype(dtype)
    idx = (rng.integers(-4, n_src + 4, n) - row_offset).astype(np.int32)
    idx[:20_000] = 17 - row_offset                       # a hot row
    gout = rng.standard_normal((n, W) if W > 1 else n).astype(dtype)
    # the adjoint: grad_src[idx + off] += grad_out in the scatter's fixed order, from zero
    z = np.zeros((n_src, W if W > 1 else 1), dtype)
    want, _ = oracle.det_scatter_add_rows(z, idx, gout.reshape(n, -1), row_offset=row_offset)
    want = want.reshape(src.shape)
    want_fwd = oracle.det_gather_rows(src, idx, row_offset=row_offset)
    grads = set()
    for _ in range(3):
        s = torch.from_numpy(src).cuda().requires_grad_(True)
        out = autograd.gather(s, torch.from_numpy(idx).cuda(), row_offset=row_offset)
        assert np.array_equal(_bits(out.detach().cpu().numpy()), _bits(want_fwd))
        out.backward(torch.from_numpy(gout).cuda())
        g = s.grad.cpu().numpy()
        assert np.array_equal(_bits(g), _bits(want))
        grads.add(g.tobytes())
    assert len(grads) == 1


def test_gather_backward_close_to_torch(ag):
    # against torch's own (CPU) gather backward: equal up to rounding order
    autograd, _ = ag
    rng = np.random.default_rng(80)
    src = rng.standard_normal((1000, 8))
    idx = rng.integers(0, 1000, 50_000).astype(np.int32)
    gout = rng.standard_normal((50_000, 8))
    s = torch.from_numpy(src).cuda().requires_grad_(True)
    autograd.gather(s, torch.from_numpy(idx).cuda()).backward(torch.from_numpy(gout).cuda())
    sc = torch.from_numpy(src).requires_grad_(True)
    sc[torch.from_numpy(idx).long()].backward(torch.from_numpy(gout))
    assert torch.allclose(s.grad.cpu(), sc.grad, rtol=0, atol=1e-12)
