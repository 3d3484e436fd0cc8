"""Seeded random shapes through every kernel path, against the oracle.

Each case draws a ragged shape (N and K multiples of 8, as TMA needs) and
one tuning configuration: one-CTA tiles of each width, split-K over a
cluster, CTA pairs with 256 x 256 or 128 x 128 tiles, stream-K through a
workspace, or the planner's own choice, with fp16 or fp32 output.  The
whole product is compared element by element with the oracle.  A second set
accumulates into C's values (C += A B) the same way.
"""
import numpy as np
import pytest

import oracle
import parity
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import draw, make_inputs

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

CONFIGS = [
    {},
    dict(cta_group=1),
    dict(cta_group=1, tile_n=64),
    dict(cta_group=1, tile_n=256),
    dict(split=2),
    dict(split=3, tile_n=64),
    dict(split=4),
    dict(cta_group=2),
    dict(cta_group=2, tile_k=64),
    dict(cta_group=2, tile_n=128),
    dict(cta_group=2, stream_k=2),
    dict(cta_group=2, tile_n=128, stream_k=2),
    dict(cta_group=1, stream_k=2),
]


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    M = int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 100))
    K = 8 * int(rng.integers(1, 300))
    cfg = CONFIGS[i % len(CONFIGS)]
    out_dtype = int(rng.integers(0, 2))
    return M, N, K, cfg, out_dtype


CASES = [draw_case(i) for i in range(40)]


@pytest.fixture(autouse=True)
def _clean_state():
    tc.gemm_f16_set_config()
    yield
    tc.gemm_f16_set_config()
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0, f"a device wait gave up (site {site})"


@pytest.mark.parametrize("M,N,K,cfg,out_dtype", CASES,
                         ids=[f"{M}x{N}x{K}-{'-'.join(f'{k}{v}' for k, v in cfg.items()) or 'plan'}-o{o}"
                              for M, N, K, cfg, o in CASES])
def test_random_shape(M, N, K, cfg, out_dtype):
    try:
        tc.gemm_f16_set_config(**cfg)
        plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
    except tc.GemmError:
        # the configuration does not fit this shape (e.g. a split longer than K):
        # the planner's own choice runs instead
        tc.gemm_f16_set_config()
        plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=M + K, seed_b=N + K)
    ws = tc.workspace(M, N, K, out_dtype) if plan["workspace_bytes"] > 0 else None
    dt = torch.float16 if out_dtype == 0 else torch.float32
    c = tc.matmul(a.cuda(), b.cuda(), out_dtype=dt, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.as_values(oracle.gemm(a.numpy(), b.numpy(), out_dtype), out_dtype)
    parity.check(c.cpu().double().numpy(), ref, K, out_dtype, f"{M}x{N}x{K} {cfg} plan {plan}")


ACC_CASES = [draw_case(100 + i) for i in range(24)]


@pytest.mark.parametrize("M,N,K,cfg,out_dtype", ACC_CASES,
                         ids=[f"acc-{M}x{N}x{K}-{'-'.join(f'{k}{v}' for k, v in cfg.items()) or 'plan'}-o{o}"
                              for M, N, K, cfg, o in ACC_CASES])
def test_random_shape_accumulate(M, N, K, cfg, out_dtype):
    """C += A B into C's values (gemm_f16_acc, no workspace) on the same kind
    of random shapes and configurations."""
    try:
        tc.gemm_f16_set_config(**cfg)
        tc.gemm_f16_plan(M, N, K, out_dtype)
    except tc.GemmError:
        tc.gemm_f16_set_config()
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=M + 2 * K, seed_b=N + 3 * K)
    c0 = draw((M, N), ("normal", 4.0), M + N)
    c0 = c0 if out_dtype == 0 else c0.float()
    c = c0.cuda()
    tc.matmul_acc(a.cuda(), b.cuda(), c)
    torch.cuda.synchronize()
    ref = oracle.as_values(oracle.gemm_acc(a.numpy(), b.numpy(), c0.numpy(), out_dtype), out_dtype)
    parity.check(c.cpu().double().numpy(), ref, K, out_dtype, f"accumulate {M}x{N}x{K} {cfg}")
