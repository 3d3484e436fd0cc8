"""The C ABI on the CPU: the library loads, exports every entry point its
header declares, rejects bad arguments before touching CUDA, and plans the
tiling the pages' arithmetic fixes.  No compute call is made here."""
import ctypes
import os
import re

import pytest

import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300 import build as tcbuild
from tensor_core_tiled_02_gb300.synthetic import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))]
# headers of the debug variants: declared only by the library of that variant
VARIANT_HEADERS = {"trace": os.path.join(ROOT, "include", "gemm_f16_trace.h"),
                   "check": os.path.join(ROOT, "include", "gemm_f16_check.h")}
PRODUCT_HEADERS = [h for h in HEADERS if h not in VARIANT_HEADERS.values()]

# status codes, as the header defines them
OK, NULL, DIM, DTYPE, ALIGN, ALIAS, CONFIG = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def lib():
    if tcbuild.needs_build():
        tcbuild.build()
    return tc.load_library()


def declared_functions(headers=None):
    """Every function the given headers (default: the product's under
    include/) declare."""
    names = set()
    for h in headers or PRODUCT_HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        text = re.sub(r"#[^\n]*", "", text)
        names.update(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(tc.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.gemm_f16_abi_version() == 2
    # the product does not carry the debug variants' entry points
    for v, h in VARIANT_HEADERS.items():
        for n in declared_functions([h]):
            assert not hasattr(lib, n), n


@pytest.mark.parametrize("variant", sorted(tcbuild.VARIANTS))
def test_debug_variants_export_the_product_abi_and_their_own(variant):
    """libtcgemm_trace.so and libtcgemm_check.so (built beside the product)
    export every product entry point, and the trace build its own."""
    path = tcbuild.variant_lib(variant)
    if not os.path.exists(path):
        tcbuild.build(variant=variant)
    vlib = ctypes.CDLL(path)
    names = declared_functions() + (declared_functions([VARIANT_HEADERS[variant]]) if variant in VARIANT_HEADERS
                                    else [])
    for n in names:
        assert hasattr(vlib, n), (variant, n)
    assert vlib.gemm_f16_abi_version() == 2


def test_add_argument_errors_before_any_cuda_call(lib):
    f = lib.add_matrices_f32
    assert f(16, 16, 16, -1, 8, None) == DIM
    assert f(16, 16, 16, 8, 6, None) == ALIGN           # rows of 24 bytes
    assert f(0, 16, 32, 8, 8, None) == NULL
    assert f(16, 24, 32, 8, 8, None) == ALIGN           # Y not 16-byte aligned
    assert f(1 << 20, 1 << 30, (1 << 20) + 64, 8, 8, None) == ALIAS   # Z partly over X
    assert f(0, 0, 0, 0, 8, None) == OK                  # empty


def test_strerror_covers_every_code(lib):
    for code, name in tc.STATUS.items():
        msg = tc.strerror(code)
        assert msg and "unknown" not in msg, name
    assert "unknown" in tc.strerror(12345)


def _call(lib, A=16, B=4096, C=1 << 20, M=128, N=128, K=64, dt=0):
    return lib.gemm_f16(A, B, C, M, N, K, dt, None)


def test_argument_errors_before_any_cuda_call(lib):
    assert _call(lib, dt=2) == DTYPE
    assert _call(lib, dt=-1) == DTYPE
    assert _call(lib, M=-1) == DIM
    assert _call(lib, N=-8) == DIM
    assert _call(lib, K=-8) == DIM
    # tile ids must fit an int for the narrowest tile, 128 x 64: 2^16 x 2^15 of them do not
    assert _call(lib, M=1 << 23, N=1 << 21) == DIM
    plan = tc.GemmPlan()
    assert lib.gemm_f16_plan(1 << 23, 1 << 21, 64, 0, 152, ctypes.byref(plan)) == DIM
    assert lib.gemm_f16_plan(1 << 23, 1 << 20, 64, 0, 152, ctypes.byref(plan)) == 0
    assert _call(lib, C=0) == NULL
    assert _call(lib, A=0) == NULL
    assert _call(lib, B=0) == NULL
    assert _call(lib, A=18) == ALIGN            # not 16-byte aligned
    assert _call(lib, C=1 << 20 | 8) == ALIGN
    assert _call(lib, N=100) == ALIGN           # row of B not a multiple of 16 bytes
    assert _call(lib, K=60) == ALIGN
    # C overlapping A: A spans [1 MiB, 1 MiB + 128*64*2)
    assert _call(lib, A=1 << 20, B=1 << 30, C=(1 << 20) + 4096) == ALIAS
    assert _call(lib, A=1 << 30, B=(1 << 20) + 64, C=1 << 20) == ALIAS
    # adjacent but not overlapping is fine up to the CUDA step; check only the
    # host arithmetic here by making another argument fail first
    assert _call(lib, A=1 << 20, B=1 << 30, C=(1 << 20) + 128 * 64 * 2, dt=5) == DTYPE


def test_empty_problems_are_noops(lib):
    # nothing is read or written: no CUDA call, success, even with NULL pointers
    assert lib.gemm_f16(0, 0, 0, 0, 128, 64, 0, None) == OK
    assert lib.gemm_f16(0, 0, 0, 128, 0, 64, 1, None) == OK


def test_plan_matches_the_tiling_arithmetic(lib):
    """Sequential steps = K / tile_k for each workload; one CTA (or CTA pair)
    per output tile; tiles = ceil(M/tile_m) * ceil(N/tile_n)."""
    # sequential steps of 64 (one CTA per tile, or the small kernel's K blocks)
    # or 128 (CTA pairs) along K
    want_k_steps = {"gemm_256": 4, "gemm_4096": 32, "gemm_8192": 64, "skinny": 128, "long_k": 256}
    for name, w in WORKLOADS.items():
        if w.kind != "gemm":
            continue
        p = tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, num_sms=152)
        assert p["k_steps"] == want_k_steps[name] == w.K // p["tile_k"]
        assert p["tile_k"] == 64 * p["cta_group"]
        assert (p["tile_m"], p["tile_n"]) in ({1: [(128, 64), (128, 128), (128, 256), (8, 64), (16, 64), (32, 64)],
                                                2: [(256, 256), (128, 128)]}[p["cta_group"]])
        assert p["tiles_m"] == -(-w.M // p["tile_m"]) and p["tiles_n"] == -(-w.N // p["tile_n"])
        assert p["num_tiles"] == p["tiles_m"] * p["tiles_n"]
        if p["cta_group"] == 2:  # one cluster of two CTAs per pair tile, persistent
            assert p["grid"] == 2 * min(p["num_tiles"], 76) and p["split"] == 1
        elif p["split"] == 1:
            assert p["grid"] == min(p["num_tiles"], 152)
        else:  # one tile per cluster of `split` CTAs
            assert p["grid"] == p["num_tiles"] * p["split"] <= 152
        assert 1 <= p["stages"] <= 8 and p["release"] < p["stages"]
        assert p["slots"] == p["stages"] + p["release"]
        assert p["smem_bytes"] <= 232448
    # the 256^3 case goes to the small kernel: 32 x 4 tiles of 8 x 64 on 128
    # CTAs, 4 K blocks of 64; on CTA pairs, 2 x 2 tiles of 128 x 128 (64 rows
    # per SM) with 2 K steps of 128; on single CTAs, the pages' tiling: 4 K
    # steps of 64
    p = tc.gemm_f16_plan(256, 256, 256, 0, num_sms=152)
    assert (p["tiles_m"], p["tiles_n"], p["tile_m"], p["tile_n"], p["k_steps"], p["cta_group"], p["grid"]) == \
        (32, 4, 8, 64, 4, 1, 128)
    assert p["tmem_cols"] == 32
    try:
        tc.gemm_f16_set_config(cta_group=2, tile_n=128)
        p = tc.gemm_f16_plan(256, 256, 256, 0, num_sms=152)
        assert (p["tiles_m"], p["tiles_n"], p["tile_m"], p["tile_n"], p["k_steps"], p["cta_group"], p["grid"]) == \
            (2, 2, 128, 128, 2, 2, 8)
        assert p["tmem_cols"] == 128
        tc.gemm_f16_set_config(cta_group=1)
        p = tc.gemm_f16_plan(256, 256, 256, 0, num_sms=152)
        assert (p["tiles_m"], p["tiles_n"], p["tile_n"], p["k_steps"], p["cta_group"]) == (2, 2, 128, 4, 1)
    finally:
        tc.gemm_f16_set_config()
    # one-CTA tiles once the 128 x 128 tiles outnumber the pairs
    p = tc.gemm_f16_plan(1280, 1024, 256, 0, num_sms=152)
    assert (p["cta_group"], p["tile_m"], p["num_tiles"], p["grid"]) == (1, 128, 80, 80)
    # the big square problem takes 256 x 256 tiles on CTA pairs
    p = tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152)
    assert (p["cta_group"], p["tile_m"], p["tile_n"], p["num_tiles"], p["grid"]) == (2, 256, 256, 1024, 152)
    assert (p["tile_k"], p["k_steps"], p["slots"]) == (128, 64, 3)
    # long K: 64 pair tiles in one wave
    p = tc.gemm_f16_plan(2048, 2048, 32768, 1, num_sms=152)
    assert (p["cta_group"], p["num_tiles"], p["split"], p["grid"]) == (2, 64, 1, 128)
    # without pairs: 128 wide tiles in one wave beat 256 narrow ones in two
    try:
        tc.gemm_f16_set_config(cta_group=1)
        p = tc.gemm_f16_plan(2048, 2048, 32768, 1, num_sms=152)
        assert (p["tile_n"], p["num_tiles"], p["split"], p["grid"]) == (256, 128, 1, 128)
    finally:
        tc.gemm_f16_set_config()
    # skinny: 64 narrow tiles would fill under half the SMs, so two CTAs share each along K
    p = tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152)
    assert (p["tile_n"], p["num_tiles"], p["split"], p["grid"]) == (128, 64, 2, 128)


def test_cta_pair_planning(lib):
    try:
        tc.gemm_f16_set_config(cta_group=2)
        p = tc.gemm_f16_plan(600, 520, 776, 0, num_sms=152)
        assert (p["tile_m"], p["tiles_m"], p["tiles_n"], p["grid"], p["slots"], p["tile_k"]) == (256, 3, 3, 18, 3, 128)
        p = tc.gemm_f16_plan(600, 520, 200, 0, num_sms=152)       # short K keeps 64-deep steps
        assert (p["tile_k"], p["k_steps"], p["slots"]) == (64, 4, 4)
        with pytest.raises(tc.GemmError):                       # no K steps to pair on
            tc.gemm_f16_plan(256, 256, 0, 0, num_sms=152)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(cta_group=2, split=2)
        tc.gemm_f16_set_config(cta_group=2, tile_n=128)      # 128 x 128 pair tiles, 128-deep steps
        p = tc.gemm_f16_plan(600, 520, 776, 0, num_sms=152)
        assert (p["tile_m"], p["tile_n"], p["tile_k"], p["tiles_m"], p["tiles_n"], p["grid"]) == \
            (128, 128, 128, 5, 5, 50)
        tc.gemm_f16_set_config(cta_group=2, tile_n=128, tile_k=64)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_plan(600, 520, 776, 0, num_sms=152)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(cta_group=2, tile_n=64)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(cta_group=3)
        tc.gemm_f16_set_config(cta_group=2, grid=4)
        assert tc.gemm_f16_plan(1100, 1280, 264, 0, num_sms=152)["grid"] == 4
        # 128-deep pipeline steps: 64 KiB per step, three fit
        tc.gemm_f16_set_config(cta_group=2, tile_k=128)
        p = tc.gemm_f16_plan(8192, 8192, 8200, 0, num_sms=152)
        assert (p["tile_k"], p["k_steps"], p["slots"]) == (128, 65, 3)
        tc.gemm_f16_set_config(cta_group=1, tile_k=128)            # single-CTA kernel: 64 only
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(tile_k=96)
    finally:
        tc.gemm_f16_set_config()


def test_tmem_never_oversubscribed(lib):
    """No SM may hold more CTAs of one launch than 512 TMEM columns serve."""
    for cfg in ({}, dict(tile_n=64), dict(tile_n=128), dict(split=2), dict(tile_n=64, split=2), dict(cta_group=2)):
        tc.gemm_f16_set_config(**cfg)
        try:
            for M, N, K in [(128, 128, 64), (256, 1024, 2048), (8192, 8192, 8192), (128, 8192, 8192)]:
                try:
                    p = tc.gemm_f16_plan(M, N, K, 0, num_sms=152)
                except tc.GemmError as e:  # e.g. a forced split longer than K
                    assert e.code == CONFIG
                    continue
                ctas_per_sm = 233472 // (p["smem_bytes"] + 1024)
                assert ctas_per_sm * p["tmem_cols"] <= 512, (cfg, M, N, K, p)
        finally:
            tc.gemm_f16_set_config()


def test_split_k_planning(lib):
    try:
        # few tiles, long K: as many CTAs per tile as fit, at most 8, >= 16 steps each
        p = tc.gemm_f16_plan(128, 128, 65536, 0, num_sms=152)
        assert (p["split"], p["grid"]) == (8, 8)
        p = tc.gemm_f16_plan(128, 128, 1024, 0, num_sms=152)   # 16 K steps: no split
        assert p["split"] == 1
        p = tc.gemm_f16_plan(128, 128, 2048, 0, num_sms=152)   # 32 K steps: 2 CTAs
        assert p["split"] == 2
        # the other ranks' fp32 partial must fit their ring: 64 KiB at tile_n 128,
        # 128 KiB at tile_n 256 (three 48 KiB buffers)
        tc.gemm_f16_set_config(split=2, stages=1)
        p = tc.gemm_f16_plan(128, 1024, 8192, 0, num_sms=152)
        assert p["slots"] * (16384 + 128 * p["tile_n"]) >= 128 * p["tile_n"] * 4
        tc.gemm_f16_set_config(split=4, tile_n=256)
        p = tc.gemm_f16_plan(256, 512, 4096, 1, num_sms=152)
        assert (p["split"], p["grid"]) == (4, 16) and p["slots"] >= 3
        tc.gemm_f16_set_config(split=4)
        with pytest.raises(tc.GemmError) as e:                  # fewer K steps than CTAs
            tc.gemm_f16_plan(128, 128, 192, 0, num_sms=152)
        assert e.value.code == CONFIG
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(split=9)
        tc.gemm_f16_set_config(split=1)
        assert tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152)["split"] == 1
    finally:
        tc.gemm_f16_set_config()


# clusters of 1 .. 8 CTAs (one per SM) a 152-SM GB300 holds at once
RESIDENT = {1: 152, 2: 76, 3: 46, 4: 36, 5: 28, 6: 23, 7: 15, 8: 15}


def test_split_k_clusters_all_fit_at_once(lib):
    """Split-K clusters must all be resident together (one wave); the split is
    lowered until they are.  Spot checks, then an invariant over many shapes."""
    p = tc.gemm_f16_plan(128, 2048, 8192, 0, num_sms=152)   # 16 tiles: 8 ranks would need 16 clusters of 8
    assert (p["num_tiles"], p["split"], p["grid"]) == (16, 6, 96)
    p = tc.gemm_f16_plan(768, 2048, 4096, 0, num_sms=152)   # 48 clusters of 3 would not fit: 2 ranks
    assert (p["tile_n"], p["num_tiles"], p["split"], p["grid"]) == (256, 48, 2, 96)
    for M in (64, 128, 256, 384, 512, 768, 1024, 1280):
        for N in (256, 512, 1024, 2048, 4096, 8192):
            for K in (2048, 8192, 32768):
                p = tc.gemm_f16_plan(M, N, K, 0, num_sms=152)
                if p["split"] > 1:
                    assert p["num_tiles"] <= RESIDENT[p["split"]], (M, N, K, p)


def test_wide_tiles_to_split_k(lib):
    """128 x 128 tiles that would run unsplit on over half the SMs give way to
    128 x 256 tiles split along K (each CTA loads 3/4 of the bytes)."""
    p = tc.gemm_f16_plan(512, 4096, 8192, 0, num_sms=152)
    assert (p["cta_group"], p["tile_n"], p["num_tiles"], p["split"], p["grid"]) == (1, 256, 64, 2, 128)
    p = tc.gemm_f16_plan(256, 8192, 8192, 0, num_sms=152)
    assert (p["cta_group"], p["tile_n"], p["num_tiles"], p["split"], p["grid"]) == (1, 256, 64, 2, 128)
    # short K: nothing to split, the narrow tiles stay
    p = tc.gemm_f16_plan(1280, 1024, 256, 0, num_sms=152)
    assert (p["tile_n"], p["split"]) == (128, 1)


def test_plan_ragged_and_degenerate(lib):
    # small problems: 128 x 128 tiles on CTA pairs with 128-deep steps
    p = tc.gemm_f16_plan(300, 392, 520, 0, num_sms=152)
    assert (p["cta_group"], p["tiles_m"], p["tiles_n"], p["k_steps"], p["grid"]) == (2, 3, 4, 5, 24)
    # the smallest: the small kernel, one CTA of 8 x 64
    p = tc.gemm_f16_plan(1, 8, 8, 1, num_sms=152)
    assert (p["cta_group"], p["tile_m"], p["tile_n"], p["num_tiles"], p["k_steps"], p["grid"]) == (1, 8, 64, 1, 1, 1)
    try:
        tc.gemm_f16_set_config(cta_group=2)
        p = tc.gemm_f16_plan(1, 8, 8, 1, num_sms=152)
        assert (p["num_tiles"], p["k_steps"], p["grid"]) == (1, 1, 2)
        tc.gemm_f16_set_config(cta_group=1)
        p = tc.gemm_f16_plan(300, 392, 520, 0, num_sms=152)
        assert (p["tiles_m"], p["tiles_n"], p["k_steps"]) == (3, 4, 9)
        p = tc.gemm_f16_plan(1, 8, 8, 1, num_sms=152)
        assert (p["num_tiles"], p["k_steps"], p["grid"]) == (1, 1, 1)
    finally:
        tc.gemm_f16_set_config()
    p = tc.gemm_f16_plan(128, 128, 0, 0, num_sms=152)
    assert p["k_steps"] == 0 and p["num_tiles"] == 1


def test_stages_clamp_and_release_rule(lib):
    """`stages` is max_concurrent_steps and `release` is delay_release: the
    ring holds stages + release buffers.  stages is clamped to the steps one
    CTA runs and must exceed release, as emit_pipeline requires."""
    try:
        tc.gemm_f16_set_config(cta_group=2)
        p = tc.gemm_f16_plan(128, 128, 256, 0, num_sms=152)  # one small pair tile: 2 steps of 128
        assert (p["cta_group"], p["stages"], p["slots"]) == (2, 2, 2)
        tc.gemm_f16_set_config(cta_group=1)
        p = tc.gemm_f16_plan(128, 128, 128, 0, num_sms=152)  # 2 steps, 1 tile
        assert (p["stages"], p["slots"]) == (2, 2)
        p = tc.gemm_f16_plan(128, 128, 64, 0, num_sms=152)   # 1 step
        assert (p["stages"], p["slots"]) == (1, 1)
        tc.gemm_f16_set_config()
        p = tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152)   # CTA pairs: 64 KiB steps
        assert (p["cta_group"], p["stages"], p["release"], p["slots"]) == (2, 3, 0, 3)
        tc.gemm_f16_set_config(cta_group=1)
        p = tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152)   # one CTA: 48 KiB steps
        assert (p["tile_n"], p["stages"], p["release"], p["slots"]) == (256, 4, 0, 4)
        # the pages' example: max_concurrent_steps=2, delay_release=1 -> 3 buffers
        tc.gemm_f16_set_config(cta_group=1, stages=2, release=1)
        p = tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152)
        assert (p["stages"], p["release"], p["slots"]) == (2, 1, 3)
        p = tc.gemm_f16_plan(128, 128, 64, 0, num_sms=152)   # clamp stops above release
        assert (p["stages"], p["slots"]) == (2, 3)
        tc.gemm_f16_set_config(cta_group=1, release=1)         # default stages: fill the ring
        p = tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152)
        assert (p["stages"], p["release"], p["slots"]) == (3, 1, 4)
        with pytest.raises(tc.GemmError) as e:
            tc.gemm_f16_set_config(stages=2, release=2)
        assert e.value.code == CONFIG
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(tile_n=192)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(stages=9)
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(stages=6, release=3)
        # a ring the shared memory cannot hold is refused at plan time
        tc.gemm_f16_set_config(tile_n=256, stages=4, release=1)
        with pytest.raises(tc.GemmError) as e:
            tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152)
        assert e.value.code == CONFIG
    finally:
        tc.gemm_f16_set_config()
    assert tc.gemm_f16_get_config()["stages"] == 0


def test_config_roundtrip(lib):
    try:
        tc.gemm_f16_set_config(tile_n=128, stages=3, release=1, grid=7, raster_group=4, cta_group=1)
        c = tc.gemm_f16_get_config()
        assert (c["tile_n"], c["stages"], c["release"], c["grid"], c["raster_group"]) == (128, 3, 1, 7, 4)
        p = tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152)
        assert (p["tile_n"], p["stages"], p["grid"], p["raster_group"]) == (128, 3, 7, 4)
    finally:
        tc.gemm_f16_set_config()


def test_plan_null_out(lib):
    assert lib.gemm_f16_plan(128, 128, 64, 0, 152, None) == NULL
    assert lib.gemm_f16_get_config(None) == NULL



def _check_plan(p, M, N, K, auto):
    """Invariants every plan must satisfy, whatever the shape or config."""
    cdiv = lambda a, b: -(-a // b)
    assert (p["tiles_m"], p["tiles_n"]) == (cdiv(M, p["tile_m"]), cdiv(N, p["tile_n"]))
    assert p["num_tiles"] == p["tiles_m"] * p["tiles_n"]
    assert p["k_steps"] == cdiv(K, p["tile_k"])
    assert p["stages"] > p["release"] >= 0 and p["slots"] == p["stages"] + p["release"]
    small = p["cta_group"] == 1 and p["tile_m"] < 128
    assert p["smem_bytes"] <= 232448 and p["threads"] == (128 if small else 192)
    # one CTA per SM at most as far as TMEM goes: no CTA ever waits on another's columns
    assert 233472 // (p["smem_bytes"] + 1024) * p["tmem_cols"] <= 512
    if p["cta_group"] == 2:
        assert p["split"] == 1 and p["grid"] % 2 == 0 and 2 <= p["grid"] <= 152
        assert (p["tile_m"], p["tile_n"], p["tmem_cols"]) in ((256, 256, 512), (128, 128, 128))
        if p["sk_tiles"] > 0:
            # stream-K owners wait on other pairs: every pair resident at once
            assert p["sk_pairs"] <= p["grid"] // 2 <= RESIDENT[2]
            assert p["dp_tiles"] + p["sk_tiles"] == p["num_tiles"]
            assert 0 < p["workspace_bytes"] <= (20 << 20) + 16384  # gemm_f16_noalloc's array holds it
        else:
            assert p["dp_tiles"] == p["num_tiles"]
    elif small:
        # the small kernel (default config only): one CTA per tile of 8, 16 or 32
        # rows by 64 columns, one wave, K <= 512 in blocks of 64 loaded at once
        assert auto and p["tile_m"] in (8, 16, 32) and (p["tile_n"], p["tile_k"], p["tmem_cols"]) == (64, 64, 32)
        assert p["grid"] == p["num_tiles"] <= 152 and p["split"] == 1 and 1 <= p["k_steps"] <= 8
        assert p["stages"] == p["slots"] == p["k_steps"] and p["sk_tiles"] == 0
        # the fewest rows that keep the tiles within one wave
        assert p["tile_m"] == 8 or cdiv(M, p["tile_m"] // 2) * p["tiles_n"] > 152
    else:
        assert p["tile_m"] == 128 and p["tile_n"] in (64, 128, 256) and p["tmem_cols"] == 2 * p["tile_n"]
        if p["split"] > 1:
            assert p["grid"] == p["num_tiles"] * p["split"] and p["split"] <= p["k_steps"]
            if auto:
                assert p["num_tiles"] <= RESIDENT[p["split"]]
        elif p["sk_tiles"] > 0:
            assert p["grid"] == p["sk_pairs"] <= 152 and p["dp_tiles"] == 0 and p["sk_tiles"] == p["num_tiles"]
        else:
            assert 1 <= p["grid"] <= 152 and p["dp_tiles"] == p["num_tiles"]


def test_plan_invariants_on_random_shapes(lib):
    """Seeded random shapes (ragged, K = 0 included) under the planner and
    under forced configurations: every plan keeps the invariants above, and a
    forced configuration either plans or is refused as GEMM_ERR_CONFIG."""
    import numpy as np

    rng = np.random.default_rng(20261202)
    configs = [({}, True), (dict(cta_group=2), False), (dict(cta_group=2, tile_n=128), False),
               (dict(cta_group=2, stream_k=2), False), (dict(cta_group=1, stream_k=2), False),
               (dict(split=2), False), (dict(split=5, tile_n=64), False), (dict(tile_n=256, stages=2), False)]
    try:
        for i in range(1500):
            M = int(rng.integers(1, 20000)) if i % 4 else int(rng.integers(1, 400))
            N = 8 * int(rng.integers(1, 2500))
            K = 8 * int(rng.integers(0, 5000)) if i % 3 else 8 * int(rng.integers(0, 64))
            cfg, auto = configs[i % len(configs)]
            tc.gemm_f16_set_config(**cfg)
            for ws in (False, True):
                try:
                    p = tc.gemm_f16_plan(M, N, K, i % 2, num_sms=152, with_workspace=ws)
                except tc.GemmError as e:
                    assert not auto and e.code == CONFIG, (M, N, K, cfg)
                    continue
                _check_plan(p, M, N, K, auto)
    finally:
        tc.gemm_f16_set_config()
