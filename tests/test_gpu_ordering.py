"""Stream order between back-to-back launches.

Every kernel here lets the next kernel in the stream start its prologue
early (programmatic dependent launch) and waits for the previous one only
just before its own first global-memory access: the producer before its
first load, the epilogue before its first store.  These tests chain launches
with no synchronisation between them, each depending on the one before, and
compare the result bit for bit with the same launches separated by a device
synchronisation (the kernels are deterministic):

  read after write   the second product reads the first one's output;
  write after read   the second launch overwrites an operand the first one
                     is still reading (a long first launch, a short second).
"""
import pytest

import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import add_inputs, make_inputs

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(autouse=True)
def _clean_state():
    tc.gemm_f16_set_config()
    yield
    tc.gemm_f16_set_config()
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0, f"a device wait gave up (site {site})"


def same_bits(x, y):
    return torch.equal(x.view(torch.int16 if x.element_size() == 2 else torch.int32),
                       y.view(torch.int16 if y.element_size() == 2 else torch.int32))


# (M, K1, N1 = K2, N2): the first product's plan, then the second's
CHAINS = {
    "pairs_stream_k": (4096, 4096, 4096, 4096),  # CTA pairs with a stream-K tail, twice
    "split_k_twice": (128, 8192, 8192, 2048),    # skinny split-K, then a split-K product of its output
    "small_pair_tiles": (640, 520, 1032, 776),   # ragged 128 x 128 tiles on CTA pairs, twice
    "one_cta_then_pair": (1280, 256, 1024, 512),  # 80 one-CTA tiles, then 40 small pair tiles
    # 12 then 6 small pair tiles: both launches prefetch their operands into L2
    # before their dependency wait, the second while the first still writes them
    "prefetching_pairs": (384, 256, 512, 256),
}


@pytest.mark.parametrize("name", list(CHAINS))
def test_read_after_write_chain(name):
    M, K1, N1, N2 = CHAINS[name]
    a, b = make_inputs(M, N1, K1, ("uniform", 1.0), ("uniform", 1.0), seed_a=11, seed_b=12)
    _, d = make_inputs(1, N2, N1, ("uniform", 1.0), ("uniform", 1.0 / 64), seed_a=13, seed_b=14)
    a, b, d = a.cuda(), b.cuda(), d.cuda()
    ws1 = tc.workspace(M, N1, K1, tc.GEMM_OUT_F16)
    ws2 = tc.workspace(M, N2, N1, tc.GEMM_OUT_F16)
    c1 = torch.empty((M, N1), dtype=torch.float16, device="cuda")
    c2 = torch.empty((M, N2), dtype=torch.float16, device="cuda")
    # separated by synchronisation
    tc.matmul(a, b, out=c1, workspace=ws1)
    torch.cuda.synchronize()
    tc.matmul(c1, d, out=c2, workspace=ws2)
    torch.cuda.synchronize()
    want1, want2 = c1.clone(), c2.clone()
    for _ in range(3):
        c1.fill_(float("nan"))
        c2.fill_(float("nan"))
        # back to back: the second launch's loads of c1 must follow the first's stores
        tc.matmul(a, b, out=c1, workspace=ws1)
        tc.matmul(c1, d, out=c2, workspace=ws2)
        torch.cuda.synchronize()
        assert same_bits(c1, want1)
        assert same_bits(c2, want2)


def test_write_after_read_chain():
    """A 4096^3 product reads x while the next launch, a 4096 x 4096 x 64
    product, overwrites x: the second launch's stores must wait for the first
    launch to finish reading."""
    M = N = K = 4096
    x, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=21, seed_b=22)
    e, f = make_inputs(M, K, 64, ("uniform", 1.0), ("uniform", 1.0), seed_a=23, seed_b=24)
    x0, b, e, f = x.cuda(), b.cuda(), e.cuda(), f.cuda()
    ws = tc.workspace(M, N, K, tc.GEMM_OUT_F16)
    xd = x0.clone()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tc.matmul(xd, b, out=c, workspace=ws)
    torch.cuda.synchronize()
    want = c.clone()
    tc.matmul(e, f, out=xd)
    torch.cuda.synchronize()
    want_x = xd.clone()
    for _ in range(3):
        xd.copy_(x0)
        c.fill_(float("nan"))
        torch.cuda.synchronize()
        tc.matmul(xd, b, out=c, workspace=ws)
        tc.matmul(e, f, out=xd)
        torch.cuda.synchronize()
        assert same_bits(c, want)
        assert same_bits(xd, want_x)


def test_blocked_add_chains():
    """z = x + y, then z = z + y in place, then x = z + z: each launch reads what
    the one before wrote, and the last overwrites an input of the first."""
    x, y = add_inputs(4096, 4096)
    x0, y = x.cuda(), y.cuda()
    xd = x0.clone()
    z = torch.empty_like(xd)
    tc.add_matrices(xd, y, out=z)
    torch.cuda.synchronize()
    tc.add_matrices(z, y, out=z)
    torch.cuda.synchronize()
    tc.add_matrices(z, z, out=xd)
    torch.cuda.synchronize()
    want_z, want_x = z.clone(), xd.clone()
    for _ in range(3):
        xd.copy_(x0)
        z.fill_(float("nan"))
        torch.cuda.synchronize()
        tc.add_matrices(xd, y, out=z)
        tc.add_matrices(z, y, out=z)
        tc.add_matrices(z, z, out=xd)
        torch.cuda.synchronize()
        assert same_bits(z, want_z)
        assert same_bits(xd, want_x)
