"""The stream-K schedule of both GEMM kernels (CTA pairs, and single CTAs),
replayed on the CPU for the plans the planner makes.

Mirrors the kernel's unit walk (data-parallel tiles c, c + clusters, ... below
dp_tiles, after cluster c's even share [S c / P, S (c+1) / P) of the
S = sk_tiles * k_steps stream-K iterations) and its owner rule (the unit that
starts a tile but does not finish it waits for the following clusters whose
shares start inside that tile).  Checked: every (tile, K step) is computed
exactly once; each partly computed tile has one owner, whose contributor set
is exactly the other units of that tile; a cluster contributes at most once
(its first unit of all, which fixes its workspace slot) and owns at most once
(its last stream-K unit), so owners wait only on contributors, which work at
the start of the launch, and nothing waits on an owner.
"""
import pytest

import tensor_core_tiled_02_gb300 as tc


def units_of(plan, c, clusters):
    KB = plan["k_steps"]
    dp = []
    t = c
    while t < plan["dp_tiles"]:
        dp.append((t, 0, KB))
        t += clusters
    sk = []
    if plan["sk_tiles"] and c < plan["sk_pairs"] and plan["sk_split"] > 0:
        # helpers: pair c < sk_tiles runs steps [0, sk_split) of shared tile c; pair
        # sk_tiles + h runs steps [sk_split, KB) of shared tiles h, h + H, ...
        dpt, S, m = plan["dp_tiles"], plan["sk_split"], plan["sk_helper_tiles"]
        H = plan["sk_pairs"] - plan["sk_tiles"]
        if c < plan["sk_tiles"]:
            sk = [(dpt + c, 0, S)]
        else:
            h = c - plan["sk_tiles"]
            sk = [(dpt + t, S, KB) for t in range(h, plan["sk_tiles"], H)]
            assert len(sk) <= m
    elif plan["sk_tiles"] and c < plan["sk_pairs"]:
        S = plan["sk_tiles"] * KB
        it, end = S * c // plan["sk_pairs"], S * (c + 1) // plan["sk_pairs"]
        while it < end:
            local, k0 = divmod(it, KB)
            k1 = min(KB, k0 + (end - it))
            sk.append((plan["dp_tiles"] + local, k0, k1))
            it += k1 - k0
    return sk + dp


def check_plan(plan):
    clusters = plan["grid"] // plan["cta_group"]
    KB = plan["k_steps"]
    cover = {}
    per_tile = {}
    for c in range(clusters):
        us = units_of(plan, c, clusters)
        for i, (t, k0, k1) in enumerate(us):
            assert 0 <= t < plan["num_tiles"] and 0 <= k0 < k1 <= KB
            for k in range(k0, k1):
                assert (t, k) not in cover, f"step {(t, k)} computed twice"
                cover[(t, k)] = c
            per_tile.setdefault(t, []).append((c, i, len(us), k0, k1))
    assert len(cover) == plan["num_tiles"] * KB, "some K step of some tile is never computed"
    S = plan["sk_tiles"] * KB
    for t, units in per_tile.items():
        if len(units) == 1:
            c, i, n, k0, k1 = units[0]
            assert (k0, k1) == (0, KB)
            continue
        owners = [u for u in units if u[3] == 0]
        assert len(owners) == 1
        oc, oi, on, _, ok1 = owners[0]
        n_sk = sum(1 for tt, _, _ in units_of(plan, oc, clusters) if tt >= plan["dp_tiles"])
        assert oi == n_sk - 1, "an owner unit must be its cluster's last stream-K unit"
        if plan["sk_split"] > 0:
            # helpers: the tile's one contributor is the helper of its index, which
            # owns nothing, and parks in the tile's own slot
            contributors = [u for u in units if u[3] > 0]
            assert len(contributors) == 1 and len(units) == 2
            hc = contributors[0][0]
            assert hc == plan["sk_tiles"] + (t - plan["dp_tiles"]) % (plan["sk_pairs"] - plan["sk_tiles"])
            assert all(k0 > 0 for tt, k0, _ in units_of(plan, hc, clusters) if tt >= plan["dp_tiles"])
            continue
        # the kernel's rule for the contributors of this tile
        tile_end = (t - plan["dp_tiles"] + 1) * KB
        q_end = oc + 1
        while q_end < plan["sk_pairs"] and S * q_end // plan["sk_pairs"] < tile_end:
            q_end += 1
        contributors = sorted(u[0] for u in units if u[3] > 0)
        assert contributors == list(range(oc + 1, q_end))
        for c, i, n, k0, k1 in units:
            if k0 > 0:
                assert i == 0, "a contributor unit must be its cluster's first unit"
                assert c < plan["sk_pairs"]


SHAPES = [(8192, 8192, 8192, 0), (4096, 4096, 4096, 0), (2048, 2048, 32768, 1), (6000, 5000, 3000, 0),
          (3072, 3072, 8192, 0), (6144, 6144, 4096, 0), (2000, 2056, 20000, 1),
          (4096, 256, 65536, 0), (20480, 20480, 1024, 0), (600, 520, 776, 0)]


SHAPES_ONE_ROW = [(128, 8192, 8192, 0), (128, 32768, 8192, 0), (100, 5000, 3000, 1), (64, 1000, 4096, 0),
                  (128, 256, 65536, 1), (1, 8, 1024, 0)]


def check_workspace(plan):
    if plan["sk_tiles"]:
        # partial slots: one per sharing cluster, or one per shared tile under helpers
        ctas = (plan["sk_tiles"] if plan["sk_split"] else plan["sk_pairs"]) * plan["cta_group"]
        # a fixed 16 KiB flag area (one word per epilogue warp of up to 1024 CTAs), then the partials
        assert plan["workspace_bytes"] == 1024 * 4 * 4 + ctas * 128 * 256 * 4


@pytest.mark.parametrize("M,N,K,dt", SHAPES)
@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("cg", [1, 2])
def test_stream_k_schedule(M, N, K, dt, mode, cg):
    try:
        tc.gemm_f16_set_config(cta_group=cg, stream_k=mode)
        for sms in (152, 148, 132):
            plan = tc.gemm_f16_plan(M, N, K, dt, num_sms=sms, with_workspace=True)
            assert plan["cta_group"] == cg
            if mode == 2:
                assert plan["sk_tiles"] > 0
            check_plan(plan)
            check_workspace(plan)
    finally:
        tc.gemm_f16_set_config()


@pytest.mark.parametrize("M,N,K,dt", SHAPES_ONE_ROW)
def test_stream_k_schedule_one_cta(M, N, K, dt):
    try:
        tc.gemm_f16_set_config(cta_group=1, stream_k=2)
        for sms in (152, 148, 132):
            plan = tc.gemm_f16_plan(M, N, K, dt, num_sms=sms, with_workspace=True)
            assert plan["cta_group"] == 1
            check_plan(plan)
            check_workspace(plan)
            assert plan["split"] == 1 and plan["dp_tiles"] == 0 and plan["grid"] == plan["sk_pairs"] <= sms
            # every share holds at least 16 K steps (or there is one share)
            assert plan["sk_pairs"] == 1 or plan["sk_tiles"] * plan["k_steps"] // plan["sk_pairs"] >= 16
    finally:
        tc.gemm_f16_set_config()


def test_one_cta_stream_k_is_opt_in():
    # M = 128: split-K clusters of two by default, with or without a workspace
    for ws in (False, True):
        p = tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152, with_workspace=ws)
        assert (p["cta_group"], p["tile_n"], p["split"], p["sk_tiles"], p["grid"]) == (1, 128, 2, 0, 128)
    try:
        tc.gemm_f16_set_config(cta_group=1, stream_k=2)
        p = tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152, with_workspace=True)
        assert (p["split"], p["dp_tiles"], p["sk_tiles"], p["sk_pairs"], p["grid"]) == (1, 0, 64, 152, 152)
        assert p["workspace_bytes"] == 16384 + 152 * 128 * 256 * 4
        assert tc.gemm_f16_workspace_size(128, 8192, 8192, 0, num_sms=152) == p["workspace_bytes"]
        # without a workspace the knob has nothing to work with
        p = tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152, with_workspace=False)
        assert p["sk_tiles"] == 0 and p["workspace_bytes"] > 0
        # an explicit split keeps the clusters
        tc.gemm_f16_set_config(cta_group=1, stream_k=2, split=2)
        assert tc.gemm_f16_plan(128, 8192, 8192, 0, num_sms=152, with_workspace=True)["sk_tiles"] == 0
    finally:
        tc.gemm_f16_set_config()


@pytest.mark.parametrize("M,N,K,dt,helpers", [(2048, 2048, 32768, 1, 11), (2000, 1800, 16000, 1, 11),
                                              (2048, 1792, 16384, 0, 19)])
def test_helpers_take_a_single_wave_more_than_half_full(M, N, K, dt, helpers):
    """R tiles on P pairs with P / 2 < R < P and no other wave: the tiles run
    their first sk_split steps on R pairs, the idle pairs run the rest, up to
    m tiles each, with 10 % slack; the wave is at least 5 % shorter."""
    p = tc.gemm_f16_plan(M, N, K, dt, num_sms=152, with_workspace=True)
    R, KB, S, m = p["sk_tiles"], p["k_steps"], p["sk_split"], p["sk_helper_tiles"]
    P = 76
    assert p["cta_group"] == 2 and R == p["num_tiles"] and P // 2 < R < P and p["dp_tiles"] == 0
    assert m == -(-R // (P - R)) and KB - S == int(0.9 * KB / (m + 1)) >= 8
    assert p["sk_pairs"] - R == helpers == -(-R // m) and p["sk_pairs"] <= P
    assert S * 100 <= KB * 95 and m * (KB - S) <= S
    assert p["workspace_bytes"] == 16384 + 2 * R * 128 * 256 * 4
    check_plan(p)
    # without a workspace the wave runs whole
    q = tc.gemm_f16_plan(M, N, K, dt, num_sms=152, with_workspace=False)
    assert q["sk_tiles"] == 0 and q["sk_split"] == 0


@pytest.mark.parametrize("M,N,K,helpers", [(6144, 6144, 4096, True), (1024, 8192, 8192, True),
                                           (3072, 3072, 8192, False), (2048, 4096, 4096, False)])
def test_helpers_after_full_waves(M, N, K, helpers):
    """After full waves, a last wave more than half full takes helpers by the
    same rule (at most 8 tiles a helper, at least 8 steps a helper unit, the
    wave at least 5 % shorter); the full waves run data-parallel after the
    shared units, on every pair.  3072 x 3072 would need 9 tiles a helper,
    2048 x 4096 x 4096 helper units of 5 steps: both stay data-parallel."""
    p = tc.gemm_f16_plan(M, N, K, 0, num_sms=152, with_workspace=True)
    P, KB, T = 76, p["k_steps"], p["num_tiles"]
    R = T % P
    assert p["cta_group"] == 2 and T > P and P // 2 < R
    if not helpers:
        assert p["sk_tiles"] == 0 and p["dp_tiles"] == T
        return
    m = -(-R // (P - R))
    assert (p["sk_tiles"], p["dp_tiles"], p["sk_helper_tiles"]) == (R, T - R, m)
    assert KB - p["sk_split"] == int(0.9 * KB / (m + 1)) >= 8 and m <= 8
    assert p["sk_pairs"] == R + -(-R // m) <= P and p["grid"] == 2 * P
    assert p["workspace_bytes"] == 16384 + 2 * R * 128 * 256 * 4
    check_plan(p)
    check_workspace(p)


def test_schedules_of_random_shapes():
    """Every stream-K schedule the planner makes for 400 seeded random shapes
    (M, N, K up to 12 288, both output types, three SM counts, with the
    workspace) covers each (tile, K step) once and keeps the owner and
    contributor rules: parts, even shares, helpers alone or after full
    waves, and one-CTA plans."""
    import numpy as np

    rng = np.random.default_rng(2024)
    kinds = set()
    for _ in range(400):
        M = int(rng.integers(1, 12289))
        N = 8 * int(rng.integers(1, 1537))
        K = 8 * int(rng.integers(1, 1537))
        dt = int(rng.integers(0, 2))
        sms = int(rng.choice([152, 148, 132]))
        p = tc.gemm_f16_plan(M, N, K, dt, num_sms=sms, with_workspace=True)
        check_plan(p)
        check_workspace(p)
        if p["sk_tiles"]:
            kinds.add(("helpers" if p["sk_split"] else "shares") + (" after waves" if p["dp_tiles"] else " alone"))
    assert {"shares after waves", "helpers alone", "helpers after waves"} <= kinds, kinds
