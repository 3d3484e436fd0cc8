"""Parity of the CUDA path with the CPU oracle, element by element.

Small and mid-size problems (several tiles, ragged tails in M, N and K) are
checked whole; the five workloads at full size, in the launch configuration
the bench times, on sampled rows and elements the oracle computes one by one.
Bit-exact properties (all-ones, identity, permutation, determinism, zero
padding) are checked where the arithmetic makes them exact.
"""
import numpy as np
import pytest

import oracle
import parity
import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300.synthetic import WORKLOADS, draw, make_inputs, workload_inputs

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


def gpu_gemm(a, b, out_dtype):
    """Run the CUDA path on CPU fp16 tensors; return the result on the CPU."""
    a_d = a.cuda()
    b_d = b.cuda()
    c = tc.matmul(a_d, b_d, out_dtype=torch.float16 if out_dtype == 0 else torch.float32)
    torch.cuda.synchronize()
    return c.cpu()


def values(c):
    return c.double().numpy()


def oracle_rows(a, b, out_dtype, rows=None):
    c = oracle.gemm(a.numpy(), b.numpy(), out_dtype, rows=rows)
    return oracle.as_values(c, out_dtype)


def check_full(a, b, out_dtype, what):
    c = gpu_gemm(a, b, out_dtype)
    ref = oracle_rows(a, b, out_dtype)
    return parity.check(values(c), ref, a.shape[1], out_dtype, what), c


# ---- whole-matrix parity ------------------------------------------------------


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_workload_256_whole(out_dtype):
    w = WORKLOADS["gemm_256"]
    a, b = workload_inputs(w)
    check_full(a, b, out_dtype, "gemm_256")


RAGGED = [(300, 392, 520), (129, 136, 72), (1, 8, 8), (127, 264, 1000), (515, 1000, 64), (64, 2056, 200)]


@pytest.mark.parametrize("M,N,K", RAGGED)
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_ragged_shapes(M, N, K, out_dtype):
    a, b = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.5), seed_a=M, seed_b=N + K)
    check_full(a, b, out_dtype, f"ragged {M}x{N}x{K}")


# every ring the shared memory holds: 8 buffers at tile_n 64, 6 at 128, 4 at 256
MAX_SLOTS = {64: 8, 128: 6, 256: 4}
VARIANTS = [dict(tile_n=t, stages=s, release=r)
            for t in (64, 128, 256) for s in range(1, 9) for r in (0, 1, 2)
            if r < s and s + r <= MAX_SLOTS[t] and (t != 64 or s in (1, 3, 8))]


@pytest.mark.parametrize("cfg", VARIANTS, ids=lambda c: f"n{c['tile_n']}s{c['stages']}r{c['release']}")
def test_pipeline_variants(cfg):
    """Every tile shape, ring depth and release depth the tuner may pick."""
    tc.gemm_f16_set_config(**cfg)
    a, b = make_inputs(300, 520, 776, ("uniform", 1.0), ("uniform", 1.0), seed_a=5, seed_b=6)
    for out_dtype in (0, 1):
        check_full(a, b, out_dtype, f"variant {cfg} out {out_dtype}")


@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_persistent_many_tiles_per_cta(tile_n):
    """A handful of CTAs each walk many tiles: the ring and both TMEM
    accumulators wrap many times across tile boundaries."""
    tc.gemm_f16_set_config(tile_n=tile_n, grid=3, raster_group=3)
    a, b = make_inputs(1100, 1024, 264, ("uniform", 1.0), ("uniform", 1.0), seed_a=9, seed_b=10)
    check_full(a, b, 0, f"persistent tile_n={tile_n}")


SPLITS = [(2, 128, 0), (2, 128, 1), (2, 256, 1), (3, 128, 0), (4, 128, 1), (8, 128, 0), (5, 256, 0), (2, 64, 0),
          (2, 64, 1), (3, 64, 1)]


@pytest.mark.parametrize("split,tile_n,out_dtype", SPLITS)
def test_split_k(split, tile_n, out_dtype):
    """Split-K through a cluster: K steps shared unevenly (47 steps), ragged
    M, N and K; partials meet through distributed shared memory, pushed by
    bulk copy between two ranks, pulled by the owner for more (with BN = 64
    and fp16 out, one rank of a pair owns no chunk at all)."""
    tc.gemm_f16_set_config(split=split, tile_n=tile_n)
    a, b = make_inputs(200, 520, 2984, ("normal", 1.0), ("normal", 1.0), seed_a=split, seed_b=tile_n)
    check_full(a, b, out_dtype, f"split {split} tile_n {tile_n}")


PAIR_VARIANTS = ([dict(cta_group=2, tile_k=64, stages=s, release=r) for s, r in [(1, 0), (2, 1), (3, 0), (4, 2), (6, 0)]]
                 + [dict(cta_group=2, tile_k=128, stages=s, release=r) for s, r in [(1, 0), (2, 1), (3, 0)]]
                 + [dict(cta_group=2, tile_n=128, stages=s, release=r) for s, r in [(1, 0), (2, 1), (3, 0), (4, 2),
                                                                                   (6, 0)]])


@pytest.mark.parametrize("cfg", PAIR_VARIANTS,
                         ids=lambda c: f"pair{c.get('tile_n', 256)}_k{c.get('tile_k', 128 if 'tile_n' in c else 64)}"
                                       f"_s{c['stages']}r{c['release']}")
def test_cta_pair_variants(cfg):
    """Tiles on a CTA pair (cta_group::2), 256 x 256 (128 rows per SM) and
    128 x 128 (64 rows per SM, folded over the TMEM lanes): ragged M (half a
    pair tile past the edge), N and K, every ring depth and release depth."""
    tc.gemm_f16_set_config(**cfg)
    a, b = make_inputs(600, 520, 776, ("uniform", 1.0), ("uniform", 1.0), seed_a=7, seed_b=8)
    for out_dtype in (0, 1):
        check_full(a, b, out_dtype, f"pair {cfg} out {out_dtype}")


def test_cta_pair_persistent_and_tiny():
    """Two pairs walk 20 pair tiles (both TMEM accumulators wrap); then a
    problem smaller than one pair tile."""
    tc.gemm_f16_set_config(cta_group=2, grid=4, raster_group=2)
    a, b = make_inputs(1100, 1280, 264, ("normal", 1.0), ("normal", 1.0), seed_a=3, seed_b=4)
    check_full(a, b, 0, "pair persistent")
    tc.gemm_f16_set_config(cta_group=2, tile_k=128, grid=4, raster_group=2)
    check_full(a, b, 1, "pair persistent, 128-deep steps")
    for tk in (64, 128):
        tc.gemm_f16_set_config(cta_group=2, tile_k=tk)
        a, b = make_inputs(64, 72, 40, ("normal", 1.0), ("normal", 1.0), seed_a=5, seed_b=6)
        check_full(a, b, 1, f"pair tiny, step {tk}")


def test_small_pair_tiles_persistent_and_exact():
    """128 x 128 pair tiles: four pairs walk 54 tiles (both TMEM accumulators
    wrap many times); all-ones and identity products are exact bit for bit."""
    tc.gemm_f16_set_config(cta_group=2, tile_n=128, grid=8, raster_group=3)
    plan = tc.gemm_f16_plan(1100, 760, 600, 0)
    assert (plan["tile_m"], plan["tile_n"], plan["num_tiles"], plan["grid"]) == (128, 128, 54, 8)
    a, b = make_inputs(1100, 760, 600, ("normal", 1.0), ("normal", 1.0), seed_a=41, seed_b=42)
    check_full(a, b, 0, "small pair tiles, persistent")
    tc.gemm_f16_set_config(cta_group=2, tile_n=128)
    ones_a = torch.ones((200, 32768), dtype=torch.float16, device="cuda")
    ones_b = torch.ones((32768, 136), dtype=torch.float16, device="cuda")
    c = tc.matmul(ones_a, ones_b, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bool((c == 32768).all())
    x, _ = make_inputs(190, 8, 264, ("uniform", 1.0), ("uniform", 1.0), seed_a=43, seed_b=44)
    eye = torch.eye(264, dtype=torch.float16)
    c = gpu_gemm(x, eye, 0)
    assert torch.equal(c.view(torch.int16), x.view(torch.int16))


def ws_gemm(a, b, out_dtype, ws):
    a_d, b_d = a.cuda(), b.cuda()
    c = tc.matmul(a_d, b_d, out_dtype=torch.float16 if out_dtype == 0 else torch.float32, workspace=ws)
    torch.cuda.synchronize()
    return c.cpu()


@pytest.mark.parametrize("tile_n", [256, 128])
@pytest.mark.parametrize("grid", [0, 10])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_stream_k_every_tile_shared(tile_n, grid, out_dtype):
    """stream_k 2: every tile's K iterations are shared by several pairs
    (owner plus contributors per tile), ragged M, N and K, on 256 x 256 and
    128 x 128 pair tiles."""
    tc.gemm_f16_set_config(cta_group=2, stream_k=2, grid=grid, tile_n=tile_n)
    plan = tc.gemm_f16_plan(1100, 1280, 2056, out_dtype, with_workspace=True)
    assert plan["sk_tiles"] == plan["num_tiles"] and plan["dp_tiles"] == 0
    ws = tc.workspace(1100, 1280, 2056, out_dtype)
    a, b = make_inputs(1100, 1280, 2056, ("normal", 1.0), ("normal", 1.0), seed_a=11, seed_b=12)
    c = ws_gemm(a, b, out_dtype, ws)
    parity.check(values(c), oracle_rows(a, b, out_dtype), 2056, out_dtype, f"stream-K all, grid {grid}")


@pytest.mark.parametrize("tile_n", [64, 128, 256])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_stream_k_one_cta_every_tile_shared(tile_n, out_dtype):
    """stream_k 2 on the one-CTA kernel: every tile's K iterations are dealt out
    to contiguous CTA shares (owner plus contributors through the workspace),
    several rows of tiles in the grouped raster, ragged M, N and K."""
    tc.gemm_f16_set_config(cta_group=1, stream_k=2, tile_n=tile_n)
    plan = tc.gemm_f16_plan(700, 1096, 3000, out_dtype, with_workspace=True)
    assert plan["cta_group"] == 1 and plan["sk_tiles"] == plan["num_tiles"] and plan["grid"] == plan["sk_pairs"]
    ws = tc.workspace(700, 1096, 3000, out_dtype)
    a, b = make_inputs(700, 1096, 3000, ("normal", 1.0), ("normal", 1.0), seed_a=21, seed_b=22)
    c = ws_gemm(a, b, out_dtype, ws)
    parity.check(values(c), oracle_rows(a, b, out_dtype), 3000, out_dtype, f"one-CTA stream-K, BN {tile_n}")


@pytest.mark.parametrize("M,N,K,out_dtype", [(100, 5000, 3000, 1), (1, 8, 1024, 0), (128, 256, 65536, 0),
                                             (77, 2056, 8200, 0)])
def test_stream_k_one_row_of_tiles(M, N, K, out_dtype):
    """One-CTA stream-K on a single row of tiles (ragged; up to 64 CTAs
    sharing one tile, a single share)."""
    tc.gemm_f16_set_config(cta_group=1, stream_k=2)
    plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
    assert plan["sk_tiles"] == plan["num_tiles"]
    ws = tc.workspace(M, N, K, out_dtype)
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=31, seed_b=32)
    c = ws_gemm(a, b, out_dtype, ws)
    parity.check(values(c), oracle_rows(a, b, out_dtype), K, out_dtype, f"{M}x{N}x{K} plan {plan['sk_pairs']}")


def test_stream_k_one_cta_reuse_determinism_and_exact_sums():
    """Consecutive calls on one workspace; repeated calls agree bit for bit;
    all-ones sums are exact through the partials."""
    tc.gemm_f16_set_config(cta_group=1, stream_k=2)
    ws = tc.workspace(128, 4096, 16384, 1)
    assert tc.gemm_f16_plan(128, 4096, 16384, 1, with_workspace=True)["sk_tiles"] > 0
    outs = []
    for seed in (1, 2, 1):
        a, b = make_inputs(128, 4096, 16384, ("uniform", 1.0), ("uniform", 1.0), seed_a=seed, seed_b=seed + 5)
        c = ws_gemm(a, b, 1, ws)
        parity.check(values(c), oracle_rows(a, b, 1), 16384, 1, f"one-CTA reuse seed {seed}")
        outs.append(c)
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))
    a = torch.ones((128, 16384), dtype=torch.float16, device="cuda")
    b = torch.ones((16384, 4096), dtype=torch.float16, device="cuda")
    c = tc.matmul(a, b, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert bool((c == 16384).all())


def test_stream_k_workspace_reuse_and_determinism():
    """One workspace serves consecutive calls (flags carry a per-launch value);
    repeated calls agree bit for bit."""
    tc.gemm_f16_set_config(cta_group=2, stream_k=2)
    ws = tc.workspace(1100, 1280, 2056, 1)
    outs = []
    for seed in (1, 2, 1):
        a, b = make_inputs(1100, 1280, 2056, ("uniform", 1.0), ("uniform", 1.0), seed_a=seed, seed_b=seed + 5)
        c = ws_gemm(a, b, 1, ws)
        parity.check(values(c), oracle_rows(a, b, 1), 2056, 1, f"reuse seed {seed}")
        outs.append(c)
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))


def test_stream_k_all_ones_exact():
    tc.gemm_f16_set_config(cta_group=2, stream_k=2)
    ws = tc.workspace(512, 512, 32768, 1)
    a = torch.ones((512, 32768), dtype=torch.float16, device="cuda")
    b = torch.ones((32768, 512), dtype=torch.float16, device="cuda")
    c = tc.matmul(a, b, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert bool((c == 32768).all())


def test_stream_k_workspace_errors():
    a = torch.ones((8192, 8192), dtype=torch.float16, device="cuda")
    c = torch.empty((8192, 8192), dtype=torch.float16, device="cuda")
    need = tc.gemm_f16_workspace_size(8192, 8192, 8192, 0)
    assert need > 0
    ws = torch.zeros(need + 256, dtype=torch.uint8, device="cuda")
    assert tc.gemm_f16_ws(a.data_ptr(), a.data_ptr(), c.data_ptr(), 8192, 8192, 8192, 0, ws.data_ptr(), need - 1,
                          0) == -12
    assert tc.gemm_f16_ws(a.data_ptr(), a.data_ptr(), c.data_ptr(), 8192, 8192, 8192, 0, ws.data_ptr() + 16, need,
                          0) == -4
    # no workspace: runs data-parallel, as gemm_f16
    assert tc.gemm_f16_ws(a.data_ptr(), a.data_ptr(), c.data_ptr(), 8192, 8192, 8192, 0, 0, 0, 0) == 0
    torch.cuda.synchronize()
    assert bool((c == 8192).all())


def test_split_k_is_deterministic():
    tc.gemm_f16_set_config(split=4)
    a, b = make_inputs(128, 1024, 4096, ("uniform", 1.0), ("uniform", 1.0), seed_a=1, seed_b=2)
    c1 = gpu_gemm(a, b, 1)
    c2 = gpu_gemm(a, b, 1)
    assert torch.equal(c1.view(torch.int32), c2.view(torch.int32))


def test_subnormal_and_scaled_inputs():
    # N(0,1)/64 inputs put ~0.3% of entries in the fp16 subnormal range
    a = draw((384, 512), ("normal", 1 / 64), 3)
    b = draw((512, 256), ("normal", 1 / 64), 4)
    assert ((a.abs() < 2 ** -14) & (a != 0)).any()
    check_full(a, b, 0, "subnormals")
    check_full(a, b, 1, "subnormals f32")


# ---- degenerate sizes -------------------------------------------------------------


def test_k_zero_writes_zeros():
    a = torch.zeros((200, 0), dtype=torch.float16, device="cuda")
    b = torch.zeros((0, 136), dtype=torch.float16, device="cuda")
    for dt in (torch.float16, torch.float32):
        c = torch.full((200, 136), 7.0, dtype=dt, device="cuda")
        tc.matmul(a, b, out_dtype=dt, out=c)
        torch.cuda.synchronize()
        assert not c.any()


def test_empty_outputs():
    a = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    b = torch.ones((64, 128), dtype=torch.float16, device="cuda")
    assert tc.matmul(a, b).shape == (0, 128)
    a = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    b = torch.ones((64, 0), dtype=torch.float16, device="cuda")
    assert tc.matmul(a, b).shape == (64, 0)


def test_errors_with_real_pointers():
    a = torch.ones((256, 256), dtype=torch.float16, device="cuda")
    b = torch.ones((256, 256), dtype=torch.float16, device="cuda")
    # C on top of A
    rc = tc.gemm_f16(a.data_ptr(), b.data_ptr(), a.data_ptr(), 256, 256, 256, 0, 0)
    assert rc == -5
    # misaligned pointer (2 bytes in)
    rc = tc.gemm_f16(a.data_ptr() + 2, b.data_ptr(), torch.empty_like(a).data_ptr(), 128, 128, 128, 0, 0)
    assert rc == -4


# ---- bit-exact properties on the GPU ---------------------------------------------


@pytest.mark.parametrize("K", [256, 4096, 8192, 32768])
def test_all_ones_exact(K):
    """All-ones A and B give C = K exactly (fp32 sums of ones are exact below 2^24)."""
    a = torch.ones((256, K), dtype=torch.float16, device="cuda")
    b = torch.ones((K, 256), dtype=torch.float16, device="cuda")
    for dt in (torch.float16, torch.float32):
        c = tc.matmul(a, b, out_dtype=dt)
        torch.cuda.synchronize()
        assert bool((c == K).all()), (K, dt)


def test_identity_returns_a_bit_exact():
    a = draw((384, 512), ("normal", 1.0), 11)
    a[a == 0] = 0  # -0 sums to +0, as in the oracle
    eye = torch.eye(512, dtype=torch.float16)
    c = gpu_gemm(a, eye, 0)
    assert torch.equal(c.view(torch.int16), a.view(torch.int16))
    c32 = gpu_gemm(a, eye, 1)
    assert torch.equal(c32, a.float())


def test_row_permutation_and_determinism():
    """Permuting rows of A permutes rows of C bit for bit (each element's
    K order is fixed), and two runs agree bit for bit."""
    a, b = make_inputs(640, 768, 1024, ("uniform", 1.0), ("uniform", 1.0), seed_a=21, seed_b=22)
    c1 = gpu_gemm(a, b, 1)
    c2 = gpu_gemm(a, b, 1)
    assert torch.equal(c1.view(torch.int32), c2.view(torch.int32))
    perm = torch.randperm(640, generator=torch.Generator().manual_seed(0))
    cp = gpu_gemm(a[perm].contiguous(), b, 1)
    assert torch.equal(cp.view(torch.int32), c1[perm].view(torch.int32))


def test_zero_padding_in_k_is_invariant():
    a, b = make_inputs(256, 256, 200, ("uniform", 1.0), ("uniform", 1.0), seed_a=31, seed_b=32)
    ap = torch.zeros((256, 256), dtype=torch.float16)
    ap[:, :200] = a
    bp = torch.zeros((256, 256), dtype=torch.float16)
    bp[:200] = b
    c = gpu_gemm(a, b, 1)
    cpad = gpu_gemm(ap, bp, 1)
    assert torch.equal(c.view(torch.int32), cpad.view(torch.int32))


def test_transpose_identity():
    """(A B)^T = B^T A^T, within the tolerance (the K order may differ)."""
    a, b = make_inputs(384, 256, 512, ("uniform", 1.0), ("uniform", 1.0), seed_a=41, seed_b=42)
    c = gpu_gemm(a, b, 1)
    ct = gpu_gemm(b.t().contiguous(), a.t().contiguous(), 1)
    ref = values(c).T
    parity.check(values(ct), ref, 512, 1, "transpose")


# ---- the five workloads at full size, sampled ----------------------------------


def sampled_rows(M, tile=128, n_random=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, min(tile - 1, M - 1), min(tile, M - 1), M - 1, max(M - tile, 0)}
    rnd = set(rng.integers(0, M, n_random).tolist())
    return np.array(sorted(fixed | rnd), np.int64)


@pytest.mark.parametrize("name", ["gemm_4096", "gemm_8192", "skinny", "long_k"])
def test_workload_full_size_sampled(name):
    w = WORKLOADS[name]
    a, b = workload_inputs(w)
    c = gpu_gemm(a, b, w.out_dtype)
    rows = sampled_rows(w.M)
    ref = oracle_rows(a, b, w.out_dtype, rows=rows)
    diag = parity.check(values(c)[rows], ref, w.K, w.out_dtype, f"{name} rows")
    # plus scattered single elements over the whole output
    rng = np.random.default_rng(1)
    ii = rng.integers(0, w.M, 2048)
    jj = rng.integers(0, w.N, 2048)
    e = oracle.as_values(oracle.gemm_elems(a.numpy(), b.numpy(), ii, jj, w.out_dtype), w.out_dtype)
    parity.check(values(c)[ii, jj], e, w.K, w.out_dtype, f"{name} elements")
    print(name, diag)


@pytest.mark.parametrize("name", ["gemm_4096", "gemm_8192", "long_k"])
def test_workload_full_size_stream_k(name):
    """The full-size workloads through gemm_f16_ws, as the bench times them:
    the last wave of tiles shared through the workspace (a thin wave in equal
    K parts over all pairs; long K's more than half full wave with helper
    pairs)."""
    w = WORKLOADS[name]
    assert tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, with_workspace=True)["sk_tiles"] > 0
    a, b = workload_inputs(w)
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype)
    c = ws_gemm(a, b, w.out_dtype, ws)
    plan = tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, with_workspace=True)
    # the first, middle and last row of every stream-K tile's row block (grouped
    # raster: groups of `raster_group` m-blocks, m-block fastest within a group)
    def m_block(t):
        g = plan["raster_group"]
        per = g * plan["tiles_n"]
        first = (t // per) * g
        return first + (t % per) % min(plan["tiles_m"] - first, g)

    rows = set(sampled_rows(w.M, n_random=4).tolist())
    for t in range(plan["dp_tiles"], plan["num_tiles"]):
        m0 = m_block(t) * 256
        rows.update(r for r in (m0, m0 + 127, m0 + 128, m0 + 255) if r < w.M)
    rows = np.array(sorted(rows), np.int64)
    ref = oracle_rows(a, b, w.out_dtype, rows=rows)
    parity.check(values(c)[rows], ref, w.K, w.out_dtype, f"{name} stream-K rows")
    rng = np.random.default_rng(2)
    ii = rng.integers(0, w.M, 2048)
    jj = rng.integers(0, w.N, 2048)
    e = oracle.as_values(oracle.gemm_elems(a.numpy(), b.numpy(), ii, jj, w.out_dtype), w.out_dtype)
    parity.check(values(c)[ii, jj], e, w.K, w.out_dtype, f"{name} stream-K elements")


def test_skinny_whole():
    """The memory-bound workload is small enough for the oracle to check whole:
    through gemm_f16_ws as the bench times it (split-K clusters of two, partials
    pushed between the pair), and with one-CTA stream-K over every SM."""
    w = WORKLOADS["skinny"]
    a, b = workload_inputs(w)
    plan = tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, with_workspace=True)
    assert plan["split"] == 2 and plan["sk_tiles"] == 0
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype)
    c = ws_gemm(a, b, w.out_dtype, ws)
    ref = oracle_rows(a, b, w.out_dtype)
    parity.check(values(c), ref, w.K, w.out_dtype, "skinny whole, split-K")
    tc.gemm_f16_set_config(cta_group=1, stream_k=2)
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype)
    c = ws_gemm(a, b, w.out_dtype, ws)
    parity.check(values(c), ref, w.K, w.out_dtype, "skinny whole, stream-K")


# ---- the device-side timeout path ----------------------------------------------------


def test_bounded_wait_reports_timeout_and_context_survives():
    """With the test hook set, no operand is ever loaded: the MMA warp's
    bounded wait runs out (~10 ms), the kernel winds down and reports the
    timeout, and the context stays usable for a normal call afterwards."""
    a, b = make_inputs(256, 256, 256, ("uniform", 1.0), ("uniform", 1.0))
    a_d, b_d = a.cuda(), b.cuda()
    tc.gemm_f16_set_config(inject_stall=1, wait_limit=20_000_000)
    tc.matmul(a_d, b_d)
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == -11 and site == 2, (rc, site)
    tc.gemm_f16_set_config()
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0 and site == 0
    c = tc.matmul(a_d, b_d)
    torch.cuda.synchronize()
    parity.check(values(c.cpu()), oracle_rows(a, b, 0), 256, 0, "after timeout")


# ---- extreme sizes ------------------------------------------------------------------


@pytest.mark.parametrize("M,N,K,out_dtype", [(8, 1 << 20, 64, 0), (1 << 20, 136, 72, 0), (256, 264, 1 << 17, 1)],
                         ids=["N=2^20", "M=2^20", "K=2^17"])
def test_extreme_shapes_sampled(M, N, K, out_dtype):
    """Very wide, very tall and very deep problems (the tile count, the raster
    and the fp32 accumulation length at their largest here), on sampled rows
    and scattered elements."""
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=13, seed_b=14)
    c = gpu_gemm(a, b, out_dtype)
    rows = sampled_rows(M, n_random=6)
    parity.check(values(c)[rows], oracle_rows(a, b, out_dtype, rows=rows), K, out_dtype, f"{M}x{N}x{K} rows")
    rng = np.random.default_rng(3)
    ii = rng.integers(0, M, 1024)
    jj = rng.integers(0, N, 1024)
    e = oracle.as_values(oracle.gemm_elems(a.numpy(), b.numpy(), ii, jj, out_dtype), out_dtype)
    parity.check(values(c)[ii, jj], e, K, out_dtype, f"{M}x{N}x{K} elements")


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_output_beyond_2_31_elements_sampled(out_dtype):
    """C of 65 536 x 32 776 (2^31 + 2^19 elements, 4.3 or 8.6 GB): the rows
    past element 2^31 (byte offsets past 4 and 8 GiB) are written, and read
    back by C += A.B, at the right places.  Checked on the rows around the
    2^31-element boundary, the last rows and a few random ones, copied back
    row by row; each row of C depends on the same row of A only, so the
    oracle computes those rows from A's."""
    M, N, K = 1 << 16, (1 << 15) + 8, 64
    a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=17, seed_b=18)
    dt = torch.float16 if out_dtype == 0 else torch.float32
    a_d, b_d = a.cuda(), b.cuda()
    c = tc.matmul(a_d, b_d, out_dtype=dt)
    torch.cuda.synchronize()
    edge = (1 << 31) // N
    rows = np.array(sorted({0, edge - 1, edge, edge + 1, M - 2, M - 1} |
                           set(np.random.default_rng(5).integers(0, M, 6).tolist())), np.int64)
    idx = torch.from_numpy(rows).cuda()
    got = c[idx].cpu()
    a_rows = a.numpy()[rows]
    parity.check(values(got), oracle_rows(torch.from_numpy(a_rows), b, out_dtype), K, out_dtype,
                 f"C beyond 2^31 elements, out {out_dtype}")
    tc.matmul_acc(a_d, b_d, c)
    torch.cuda.synchronize()
    got2 = c[idx].cpu()
    del c
    torch.cuda.empty_cache()
    ref2 = oracle.as_values(oracle.gemm_acc(a_rows, b.numpy(), got.numpy(), out_dtype), out_dtype)
    parity.check(values(got2), ref2, K, out_dtype, f"C += A.B beyond 2^31 elements, out {out_dtype}")


# ---- CUDA graphs ----------------------------------------------------------------------


def test_graph_capture_and_replay():
    """Launches of gemm_f16 and gemm_f16_ws captured in a CUDA graph and
    replayed give the eager results bit for bit (tensor maps and launch
    parameters are captured by value)."""
    a1, b1 = make_inputs(512, 768, 1024, ("uniform", 1.0), ("uniform", 1.0), seed_a=1, seed_b=2)
    a2, b2 = make_inputs(4096, 4096, 1024, ("uniform", 1.0), ("uniform", 1.0), seed_a=3, seed_b=4)
    a1d, b1d, a2d, b2d = a1.cuda(), b1.cuda(), a2.cuda(), b2.cuda()
    ws = tc.workspace(4096, 4096, 1024, 0)
    c1 = torch.empty((512, 768), dtype=torch.float16, device="cuda")
    c2 = torch.empty((4096, 4096), dtype=torch.float16, device="cuda")
    # eager reference (also does each device's one-time set-up outside the capture)
    tc.matmul(a1d, b1d, out=c1)
    tc.matmul(a2d, b2d, out=c2, workspace=ws)
    torch.cuda.synchronize()
    e1, e2 = c1.clone(), c2.clone()
    c1.zero_()
    c2.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            tc.matmul(a1d, b1d, out=c1)
            tc.matmul(a2d, b2d, out=c2, workspace=ws)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), e1.view(torch.int16))
    assert torch.equal(c2.view(torch.int16), e2.view(torch.int16))


def test_graph_replay_of_stream_k_waits_for_each_replays_partials():
    """One stream-K launch (the thin last wave of 4096^3 shared through the
    workspace) captured once and replayed with new operands in the same
    buffers: every replay carries the same flag value, so each owner must
    hand its consumed flags back (zero) for the next replay to wait on its
    own partials.  Each replay equals an eager call on the same operands."""
    M = N = K = 4096
    plan = tc.gemm_f16_plan(M, N, K, 0, with_workspace=True)
    assert plan["sk_tiles"] > 0
    ws = tc.workspace(M, N, K, 0)
    a_d = torch.empty((M, K), dtype=torch.float16, device="cuda")
    b_d = torch.empty((K, N), dtype=torch.float16, device="cuda")
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    a1, b1 = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=71, seed_b=72)
    a_d.copy_(a1)
    b_d.copy_(b1)
    tc.matmul(a_d, b_d, out=c, workspace=ws)  # one-time set-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tc.matmul(a_d, b_d, out=c, workspace=ws)
    for seed in (81, 82, 83):
        a, b = make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=seed, seed_b=seed + 1)
        a_d.copy_(a)
        b_d.copy_(b)
        c.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = c.clone()
        want = tc.matmul(a_d, b_d, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"replay with seed {seed}"



# ---- helper stream-K: a last wave more than half full ----------------------------


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_helper_stream_k_whole(out_dtype):
    """64 ragged pair tiles (2000 x 1800, K = 16000: 125 steps, the last one
    ragged) on the GPU's pairs: each tile's first sk_split steps run on its own
    pair, the idle pairs run the rest of several tiles each, and each tile
    meets one helper's partial.  Checked whole against the oracle, and bit for
    bit against itself on a second call (the flags are handed back)."""
    M, N, K = 2000, 1800, 16000
    plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
    assert plan["sk_split"] > 0 and plan["sk_tiles"] == 64, plan
    ws = tc.workspace(M, N, K, out_dtype)
    a, b = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), seed_a=91, seed_b=92)
    c = ws_gemm(a, b, out_dtype, ws)
    parity.check(values(c), oracle_rows(a, b, out_dtype), K, out_dtype, f"helper stream-K out {out_dtype}")
    c2 = ws_gemm(a, b, out_dtype, ws)
    bits = torch.int16 if out_dtype == 0 else torch.int32
    assert torch.equal(c.view(bits), c2.view(bits))


@pytest.mark.parametrize("M,N,K,out_dtype", [(1000, 7992, 8200, 0), (1000, 7424, 3456, 1)])
def test_helper_stream_k_after_full_waves_whole(M, N, K, out_dtype):
    """A full wave of pair tiles, then a last wave more than half full whose
    tiles take helpers (shared units first, the data-parallel wave after them
    on every pair); ragged M, N and K.  Checked whole against the oracle, and
    bit for bit against itself on a second call."""
    plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=True)
    pairs = plan["grid"] // 2
    assert plan["dp_tiles"] >= pairs and plan["sk_split"] > 0 and plan["sk_pairs"] < pairs, plan
    ws = tc.workspace(M, N, K, out_dtype)
    a, b = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), seed_a=97, seed_b=98)
    c = ws_gemm(a, b, out_dtype, ws)
    parity.check(values(c), oracle_rows(a, b, out_dtype), K, out_dtype, f"helpers after full waves, out {out_dtype}")
    c2 = ws_gemm(a, b, out_dtype, ws)
    bits = torch.int16 if out_dtype == 0 else torch.int32
    assert torch.equal(c.view(bits), c2.view(bits))


# ---- the small kernel ----------------------------------------------------------------


SMALL_SHAPES = [(256, 256, 256, 0, 8), (1, 8, 8, 1, 8), (8, 64, 64, 0, 8), (300, 264, 504, 0, 16),
                (200, 520, 504, 1, 16), (512, 512, 512, 1, 32), (64, 4096, 512, 0, 32), (37, 1000, 72, 0, 8),
                (129, 616, 448, 1, 16), (600, 376, 264, 0, 32)]


@pytest.mark.parametrize("M,N,K,out_dtype,rows", SMALL_SHAPES)
def test_small_kernel_whole(M, N, K, out_dtype, rows):
    """Problems the small kernel takes (one CTA per rows x 64 tile of C, the
    transposed MMA with M = 64, K <= 512 loaded at once), ragged in M, N and
    K: C = A.B and then C += A.B checked whole against the oracle, and the
    product bit for bit on a second call."""
    plan = tc.gemm_f16_plan(M, N, K, out_dtype)
    assert (plan["cta_group"], plan["tile_m"], plan["tile_n"]) == (1, rows, 64), plan
    a, b = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), seed_a=M, seed_b=N + K)
    a_d, b_d = a.cuda(), b.cuda()
    dt = torch.float16 if out_dtype == 0 else torch.float32
    c = tc.matmul(a_d, b_d, out_dtype=dt)
    c2 = tc.matmul(a_d, b_d, out_dtype=dt)
    torch.cuda.synchronize()
    parity.check(values(c.cpu()), oracle_rows(a, b, out_dtype), K, out_dtype, f"small {M}x{N}x{K}")
    bits = torch.int16 if out_dtype == 0 else torch.int32
    assert torch.equal(c.view(bits), c2.view(bits))
    c0 = c.cpu()
    tc.matmul_acc(a_d, b_d, c)
    torch.cuda.synchronize()
    ref = oracle.as_values(oracle.gemm_acc(a.numpy(), b.numpy(), c0.numpy(), out_dtype), out_dtype)
    parity.check(values(c.cpu()), ref, K, out_dtype, f"small {M}x{N}x{K}, C += A.B")
