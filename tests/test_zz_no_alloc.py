"""gemm_f16_noalloc: the entry point for callers that cannot allocate device
memory when they call (an allocator that must not re-enter the CUDA
allocator, a plugin handed only its buffers, latency-critical code where
cudaMalloc may synchronise the device).  Its stream-K scratch is a fixed
array in device memory, shared by all calls.

Called through the C ABI, it must give what gemm_f16_ws gives with a
caller-owned workspace, within the parity tolerance, on two calls in a row
with different operands (the second call must not see the first one's
partial tiles).  Runs alone in a fresh process or after the other tests.
"""
import ctypes

import numpy as np
import pytest

import parity
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import make_inputs

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def run_pair(lib, M, N, K, out_dtype, seed):
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=seed, seed_b=seed + 100)
    a, b = a.cuda(), b.cuda()
    dt = torch.float16 if out_dtype == 0 else torch.float32
    c_noalloc = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    c_ref = torch.empty((M, N), dtype=dt, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gemm_f16_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                              ctypes.c_void_p(c_noalloc.data_ptr()), M, N, K, out_dtype, ctypes.c_void_p(stream))
    assert rc == 0, tc.strerror(rc)
    ws = tc.workspace(M, N, K, out_dtype)
    rc = tc.gemm_f16_ws(a.data_ptr(), b.data_ptr(), c_ref.data_ptr(), M, N, K, out_dtype, ws.data_ptr(),
                        ws.numel(), stream)
    assert rc == 0, tc.strerror(rc)
    torch.cuda.synchronize()
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0, f"a device wait gave up (site {site})"
    return c_noalloc.cpu().double().numpy(), c_ref.cpu().double().numpy()


@pytest.mark.parametrize("shape,cfg", [((4096, 4096, 4096, 0), {}),
                                       ((1100, 1280, 2056, 1), dict(cta_group=2, stream_k=2)),
                                       ((128, 8192, 8192, 0), dict(cta_group=1, stream_k=2))],
                         ids=["4096_tail_stream_k", "every_tile_shared", "one_row_every_sm"])
def test_noalloc_matches_workspace_entry_on_two_calls(shape, cfg):
    lib = tc.load_library()
    M, N, K, out_dtype = shape
    try:
        tc.gemm_f16_set_config(**cfg)
        plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
        assert plan["sk_tiles"] > 0, "the problem must use the stream-K scratch"
        for seed in (1, 2):
            got, want = run_pair(lib, M, N, K, out_dtype, seed)
            assert not np.isnan(got).any()
            parity.check(got, want, K, out_dtype, f"noalloc call {seed} vs gemm_f16_ws")
    finally:
        tc.gemm_f16_set_config()


def test_noalloc_refuses_bad_arguments_like_gemm_f16():
    lib = tc.load_library()
    assert lib.gemm_f16_noalloc(None, None, None, -1, 8, 8, 0, None) == -2
    assert lib.gemm_f16_noalloc(None, None, None, 8, 8, 8, 7, None) == -3
