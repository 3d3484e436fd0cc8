"""gemm_f16_noalloc: the entry point for callers that cannot allocate device
memory when they call (an allocator that must not re-enter the CUDA
allocator, a plugin handed only its buffers, latency-critical code where
cudaMalloc may synchronise the device).  Its stream-K scratch is a fixed
array in device memory, shared by all calls.

Called through the C ABI, it must give exactly what gemm_f16_ws gives with a
caller-owned workspace (the two run the same plan, and every kernel here is
deterministic, so the outputs agree bit for bit), on two calls in a row with
different operands (the second call must not see the first one's partial
tiles), and match the oracle on sampled rows, on the first and last rows of
every stream-K tile and on scattered elements.  A plan that shares tiles
over few CTAs followed by one that shares them over many checks that the
later call's flags never read the earlier call's leftovers.  Runs alone in a
fresh process or after the other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
import parity
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import make_inputs

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def run_both(lib, a, b, M, N, K, out_dtype):
    """C through gemm_f16_noalloc and through gemm_f16_ws, same operands."""
    dt = torch.float16 if out_dtype == 0 else torch.float32
    c_noalloc = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    c_ref = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
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
    return c_noalloc.cpu(), c_ref.cpu()


def stream_k_rows(plan, M, seed):
    """Rows 0, 1, M-1, a few random ones, and the first, middle and last rows
    of the row block of every tile whose K iterations are shared (grouped
    raster: groups of raster_group m-blocks, the m-block fastest inside)."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1} | set(rng.integers(0, M, 6).tolist())
    g, tiles_m, tiles_n, tm = plan["raster_group"], plan["tiles_m"], plan["tiles_n"], plan["tile_m"]
    for t in range(plan["dp_tiles"], plan["num_tiles"]):
        per = g * tiles_n
        first = (t // per) * g
        mb = first + (t % per) % min(tiles_m - first, g)
        m0 = mb * tm
        rows.update(r for r in (m0, m0 + tm // 2 - 1, m0 + tm // 2, m0 + tm - 1) if r < M)
    return np.array(sorted(rows), np.int64)


def check_against_oracle(a, b, c, plan, M, N, K, out_dtype, seed, what):
    got = c.double().numpy()
    rows = stream_k_rows(plan, M, seed)
    ref = oracle.as_values(oracle.gemm(a.numpy(), b.numpy(), out_dtype, rows=rows), out_dtype)
    parity.check(got[rows], ref, K, out_dtype, f"{what} rows")
    rng = np.random.default_rng(seed + 7)
    ii = rng.integers(0, M, 1024)
    jj = rng.integers(0, N, 1024)
    e = oracle.as_values(oracle.gemm_elems(a.numpy(), b.numpy(), ii, jj, out_dtype), out_dtype)
    parity.check(got[ii, jj], e, K, out_dtype, f"{what} elements")


def bits(c):
    return c.view(torch.int16) if c.dtype == torch.float16 else c.view(torch.int32)


CASES = [((4096, 4096, 4096, 0), {}),
         ((1100, 1280, 2056, 1), dict(cta_group=2, stream_k=2)),
         ((128, 8192, 8192, 0), dict(cta_group=1, stream_k=2)),
         ((2000, 1800, 16000, 1), {}),
         ((1000, 7424, 3456, 1), {})]


@pytest.mark.parametrize("shape,cfg", CASES, ids=["4096_tail_stream_k", "every_tile_shared", "one_row_every_sm",
                                                  "helper_pairs", "helpers_after_a_full_wave"])
def test_noalloc_matches_workspace_entry_on_two_calls(shape, cfg):
    lib = tc.load_library()
    M, N, K, out_dtype = shape
    try:
        tc.gemm_f16_set_config(**cfg)
        plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
        assert plan["sk_tiles"] > 0, "the problem must use the stream-K scratch"
        for seed in (1, 2):
            a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=seed, seed_b=seed + 100)
            got, want = run_both(lib, a.cuda(), b.cuda(), M, N, K, out_dtype)
            assert not torch.isnan(got).any()
            assert torch.equal(bits(got), bits(want)), f"call {seed}: noalloc differs from gemm_f16_ws"
            check_against_oracle(a, b, got, plan, M, N, K, out_dtype, seed, f"noalloc call {seed}")
    finally:
        tc.gemm_f16_set_config()


def test_noalloc_few_sharing_ctas_then_many():
    """A plan sharing tiles over 10 CTAs (5 pairs), then one sharing them over
    every SM: the second call's flags lie where the first call kept nothing
    but flags, and both calls match gemm_f16_ws bit for bit and the oracle."""
    lib = tc.load_library()
    steps = [((1100, 1280, 2056, 1), dict(cta_group=2, stream_k=2, grid=10)),
             ((128, 8192, 8192, 1), dict(cta_group=1, stream_k=2))]
    counts = []
    try:
        for i, ((M, N, K, out_dtype), cfg) in enumerate(steps):
            tc.gemm_f16_set_config(**cfg)
            plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
            assert plan["sk_tiles"] > 0
            counts.append(plan["sk_pairs"] * plan["cta_group"])
            a, b = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), seed_a=40 + i, seed_b=50 + i)
            got, want = run_both(lib, a.cuda(), b.cuda(), M, N, K, out_dtype)
            assert torch.equal(bits(got), bits(want)), f"step {i}: noalloc differs from gemm_f16_ws"
            check_against_oracle(a, b, got, plan, M, N, K, out_dtype, 60 + i, f"noalloc step {i}")
    finally:
        tc.gemm_f16_set_config()
    assert counts[0] < counts[1], counts


def test_noalloc_refuses_bad_arguments_like_gemm_f16():
    lib = tc.load_library()
    assert lib.gemm_f16_noalloc(None, None, None, -1, 8, 8, 0, None) == -2
    assert lib.gemm_f16_noalloc(None, None, None, 8, 8, 8, 7, None) == -3
