"""C += A B (gemm_f16_acc): the product accumulated into what C holds,
against the oracle's accumulate form, in every kernel mode."""
import numpy as np
import pytest

import oracle
import parity
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import draw, make_inputs

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


CASES = [
    ("one CTA, ragged", (300, 392, 520), {}),
    ("split-K", (128, 1024, 4096), {}),
    ("CTA pair", (600, 520, 776), dict(cta_group=2)),
    ("CTA pair, 64-deep steps", (600, 520, 200), dict(cta_group=2)),
    ("128 x 64 tiles", (200, 136, 264), dict(tile_n=64)),
]


@pytest.mark.parametrize("name,shape,cfg", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_accumulate(name, shape, cfg, out_dtype):
    M, N, K = shape
    tc.gemm_f16_set_config(**cfg)
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=M + 1, seed_b=N + 2)
    c0 = draw((M, N), ("normal", 8.0), 7)
    c0 = c0 if out_dtype == 0 else c0.float()
    c = c0.cuda()
    tc.matmul_acc(a.cuda(), b.cuda(), c)
    torch.cuda.synchronize()
    ref = oracle.as_values(oracle.gemm_acc(a.numpy(), b.numpy(), c0.numpy(), out_dtype), out_dtype)
    parity.check(c.cpu().double().numpy(), ref, K, out_dtype, f"accumulate {name}")


def test_accumulate_with_no_k_leaves_c():
    c0 = draw((200, 136), ("normal", 1.0), 3)
    for dt in (torch.float16, torch.float32):
        c = c0.to(dt).cuda()
        tc.matmul_acc(torch.zeros((200, 0), dtype=torch.float16, device="cuda"),
                      torch.zeros((0, 136), dtype=torch.float16, device="cuda"), c)
        torch.cuda.synchronize()
        assert torch.equal(c.cpu(), c0.to(dt))


def test_two_accumulations_chain():
    """C = C0 + A1 B1, then C += A2 B2: the second call starts from the first's
    rounded result."""
    M, N, K = 256, 384, 512
    a1, b1 = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=1, seed_b=2)
    a2, b2 = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=3, seed_b=4)
    c0 = draw((M, N), ("normal", 4.0), 5).float()
    c = c0.cuda()
    tc.matmul_acc(a1.cuda(), b1.cuda(), c)
    torch.cuda.synchronize()
    mid = c.cpu().numpy().copy()
    tc.matmul_acc(a2.cuda(), b2.cuda(), c)
    torch.cuda.synchronize()
    ref1 = oracle.gemm_acc(a1.numpy(), b1.numpy(), c0.numpy(), oracle.OUT_F32)
    parity.check(mid.astype(np.float64), ref1.astype(np.float64), K, 1, "first accumulation")
    ref2 = oracle.gemm_acc(a2.numpy(), b2.numpy(), mid, oracle.OUT_F32)
    parity.check(c.cpu().double().numpy(), ref2.astype(np.float64), K, 1, "second accumulation")


def test_accumulate_refuses_aliasing():
    a = torch.ones((256, 256), dtype=torch.float16, device="cuda")
    b = torch.ones((256, 256), dtype=torch.float16, device="cuda")
    assert tc.load_library().gemm_f16_acc(a.data_ptr(), b.data_ptr(), a.data_ptr(), 256, 256, 256, 0, None) == -5
