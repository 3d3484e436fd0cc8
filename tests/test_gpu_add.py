"""The pipelined blocked add Z = X + Y on the GPU, bit for bit against the
oracle (the pages check it with assert_array_equal)."""
import numpy as np
import pytest

import oracle
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import add_inputs

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(autouse=True)
def _status():
    yield
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0, f"a device wait gave up (site {site})"


def check(x, y, z_gpu):
    want = oracle.add_f32(x.numpy(), y.numpy())
    assert np.array_equal(z_gpu.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_the_pages_workload():
    """f32[4096, 4096], both ~ U[0, 1), as the blocked-add example draws them."""
    x, y = add_inputs(4096, 4096)
    z = tc.add_matrices(x.cuda(), y.cuda())
    torch.cuda.synchronize()
    check(x, y, z)


@pytest.mark.parametrize("M,N", [(1, 4), (31, 260), (33, 256), (100, 1000), (513, 772), (4097, 4100)])
def test_ragged_shapes(M, N):
    x, y = add_inputs(M, N, 3, 4)
    z = tc.add_matrices(x.cuda(), y.cuda())
    torch.cuda.synchronize()
    check(x, y, z)


def test_special_values_and_in_place():
    rng = np.random.default_rng(5)
    xs = (rng.choice([-1.0, 1.0], (300, 512)) * np.exp2(rng.uniform(-149, 127, (300, 512)))).astype(np.float32)
    ys = (rng.choice([-1.0, 1.0], (300, 512)) * np.exp2(rng.uniform(-149, 127, (300, 512)))).astype(np.float32)
    xs[0, :6] = [np.inf, -np.inf, -0.0, 2.0 ** -149, 3.4028234663852886e38, 1.0]
    ys[0, :6] = [-np.inf, 1.0, -0.0, 2.0 ** -149, 3.4028234663852886e38, 2.0 ** -24]
    x, y = torch.from_numpy(xs), torch.from_numpy(ys)
    xd = x.cuda()
    tc.add_matrices(xd, y.cuda(), out=xd)  # in place: Z is X
    torch.cuda.synchronize()
    got = xd.cpu().numpy()
    want = oracle.add_f32(xs, ys)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_errors_with_real_pointers():
    x = torch.ones((64, 64), dtype=torch.float32, device="cuda")
    lib = tc.load_library()
    assert lib.add_matrices_f32(x.data_ptr(), x.data_ptr(), x.data_ptr() + 256, 64, 64, None) == -5
    assert lib.add_matrices_f32(x.data_ptr() + 4, x.data_ptr(), x.data_ptr(), 8, 8, None) == -4
