"""The bounds-check build's arithmetic on the CPU (no GPU).

libtcgemm_check.so (-DTCGEMM_CHECK) tests every shared-memory, Tensor Memory
and workspace access in its kernels against the allocation before making it.
Its host entry point gemm_f16_check_plan runs the same tests, on the same
arithmetic (csrc/bounds.cuh), over every access a plan's launch makes: here
every plan the planner gives must pass, and plans with a planted mistake
(a ring slot more than the shared memory holds, half the Tensor Memory, a
short workspace) must fail at the right site."""
import ctypes
import os

import numpy as np
import pytest

import tensor_core_tiled_02_gb300 as tc
from tensor_core_tiled_02_gb300 import build as tcbuild

SMEM, TMEM, WORKSPACE = 9, 10, 11


@pytest.fixture(scope="module")
def check_lib():
    path = tcbuild.variant_lib("check")
    if not os.path.exists(path):
        tcbuild.build(variant="check")
    lib = ctypes.CDLL(path)
    lib.gemm_f16_check_plan.argtypes = [ctypes.POINTER(tc.GemmPlan), ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.gemm_f16_check_plan.restype = ctypes.c_int
    return lib


def plan_struct(M, N, K, dt, ws=True, **cfg):
    tc.gemm_f16_set_config(**cfg)
    try:
        d = tc.gemm_f16_plan(M, N, K, dt, num_sms=152, with_workspace=ws)
    finally:
        tc.gemm_f16_set_config()
    p = tc.GemmPlan()
    for k, v in d.items():
        setattr(p, k, v)
    return p


def site_of(lib, p, dt):
    site = ctypes.c_int(-1)
    rc = lib.gemm_f16_check_plan(ctypes.byref(p), dt, ctypes.byref(site))
    assert (rc == 0) == (site.value == 0), (rc, site.value)
    return site.value


def test_every_planned_launch_stays_in_bounds(check_lib):
    rng = np.random.default_rng(20261203)
    configs = [{}, dict(cta_group=2), dict(cta_group=2, tile_n=128), dict(cta_group=2, stream_k=2),
               dict(cta_group=1, stream_k=2), dict(split=2), dict(split=3, tile_n=64), dict(split=2, tile_n=256),
               dict(split=8), dict(tile_n=256, stages=2, release=1), dict(tile_n=64, stages=7, release=1),
               dict(cta_group=2, tile_k=64, stages=5, release=1)]
    checked = 0
    for i in range(600):
        M = int(rng.integers(1, 20000)) if i % 4 else int(rng.integers(1, 400))
        N = 8 * int(rng.integers(1, 2500))
        K = 8 * int(rng.integers(1, 5000)) if i % 3 else 8 * int(rng.integers(1, 64))
        cfg = configs[i % len(configs)]
        for dt in (0, 1):
            try:
                p = plan_struct(M, N, K, dt, **cfg)
            except tc.GemmError:
                continue  # a forced configuration this problem refuses
            assert site_of(check_lib, p, dt) == 0, (M, N, K, dt, cfg)
            checked += 1
    assert checked > 900


@pytest.mark.parametrize("shape", [(8192, 8192, 8192, 0), (128, 8192, 8192, 0), (2048, 2048, 32768, 1),
                                   (256, 256, 256, 0), (4096, 4096, 4096, 0)])
def test_the_five_workloads_plans_stay_in_bounds(check_lib, shape):
    M, N, K, dt = shape
    assert site_of(check_lib, plan_struct(M, N, K, dt), dt) == 0


def test_planted_mistakes_are_caught(check_lib):
    # a ring slot more than the requested shared memory holds
    p = plan_struct(8192, 8192, 8192, 0)
    p.slots += 1
    p.stages += 1
    assert site_of(check_lib, p, 0) == SMEM
    # the requested shared memory short by two KiB
    p = plan_struct(8192, 8192, 8192, 0)
    p.smem_bytes -= 2048
    assert site_of(check_lib, p, 0) == SMEM
    # more ring slots than the kernel has barriers for
    p = plan_struct(256, 256, 256, 0, cta_group=2)
    p.slots = 9
    assert site_of(check_lib, p, 0) == SMEM
    # the small kernel: shared memory short by two KiB, more K blocks than it
    # holds, a CTA short of its tile, half its Tensor Memory
    p = plan_struct(256, 256, 256, 0)
    assert (p.tile_m, p.tile_n) == (8, 64)
    p.smem_bytes -= 2048
    assert site_of(check_lib, p, 0) == SMEM
    p = plan_struct(256, 256, 256, 0)
    p.k_steps = 9
    assert site_of(check_lib, p, 0) == SMEM
    p = plan_struct(256, 256, 256, 0)
    p.grid -= 1
    assert site_of(check_lib, p, 0) == SMEM
    p = plan_struct(256, 256, 256, 0)
    p.tmem_cols //= 2
    assert site_of(check_lib, p, 0) == TMEM
    # half the Tensor Memory the two accumulators need
    p = plan_struct(128, 8192, 8192, 0)
    p.tmem_cols //= 2
    assert site_of(check_lib, p, 0) == TMEM
    # a stream-K workspace one partial short, or more sharing CTAs than flags
    p = plan_struct(4096, 4096, 4096, 0)
    assert p.sk_tiles > 0
    p.workspace_bytes -= 128 * 256 * 4
    assert site_of(check_lib, p, 0) == WORKSPACE
    p = plan_struct(4096, 4096, 4096, 0)
    p.sk_pairs = 513
    assert site_of(check_lib, p, 0) == WORKSPACE
    # split-K 3 on 128 x 256 fp32 tiles parks 2 x 4 warps x 8 chunks x 4 KiB in
    # the ring: a ring of one slot cannot hold them
    p = plan_struct(128, 256, 8192, 1, split=3, tile_n=256)
    p.slots, p.stages, p.release = 1, 1, 0
    assert site_of(check_lib, p, 1) == SMEM
    # a tile no kernel has
    p = plan_struct(256, 256, 256, 0)
    p.tile_n = 96
    assert site_of(check_lib, p, 0) == SMEM


def test_check_plan_argument_errors(check_lib):
    p = plan_struct(256, 256, 256, 0)
    site = ctypes.c_int(0)
    assert check_lib.gemm_f16_check_plan(None, 0, ctypes.byref(site)) == -1
    assert check_lib.gemm_f16_check_plan(ctypes.byref(p), 0, None) == -1
    assert check_lib.gemm_f16_check_plan(ctypes.byref(p), 3, ctypes.byref(site)) == -3
