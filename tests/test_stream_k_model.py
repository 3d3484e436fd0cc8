"""The stream-K schedule of the CTA-pair kernel, replayed on the CPU for the
plans the planner makes.

Mirrors the kernel's unit walk (data-parallel tiles c, c + clusters, ... below
dp_tiles, then cluster c's even share [S c / P, S (c+1) / P) of the
S = sk_tiles * k_steps stream-K iterations) and its owner rule (the unit that
starts a tile but does not finish it waits for the following clusters whose
shares start inside that tile).  Checked: every (tile, K step) is computed
exactly once; each partly computed tile has one owner, whose contributor set
is exactly the other units of that tile; a cluster contributes at most once
(its first stream-K unit, which fixes its workspace slot) and owns at most
once (its last unit), so owners wait only on contributors, which work at the
start of the stream-K phase, and nothing waits on an owner.
"""
import pytest

import tensor_core_tiled_02_gb300 as tc


def units_of(plan, c, clusters):
    KB = plan["k_steps"]
    out = []
    t = c
    while t < plan["dp_tiles"]:
        out.append((t, 0, KB))
        t += clusters
    if plan["sk_tiles"] and c < plan["sk_pairs"]:
        S = plan["sk_tiles"] * KB
        it, end = S * c // plan["sk_pairs"], S * (c + 1) // plan["sk_pairs"]
        while it < end:
            local, k0 = divmod(it, KB)
            k1 = min(KB, k0 + (end - it))
            out.append((plan["dp_tiles"] + local, k0, k1))
            it += k1 - k0
    return out


def check_plan(plan):
    clusters = plan["grid"] // 2
    KB = plan["k_steps"]
    cover = {}
    per_tile = {}
    dp_units = {}
    for c in range(clusters):
        us = units_of(plan, c, clusters)
        dp_units[c] = sum(1 for t, _, _ in us if t < plan["dp_tiles"])
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
        assert oi == on - 1, "an owner unit must be its cluster's last"
        # the kernel's rule for the contributors of this tile
        tile_end = (t - plan["dp_tiles"] + 1) * KB
        q_end = oc + 1
        while q_end < plan["sk_pairs"] and S * q_end // plan["sk_pairs"] < tile_end:
            q_end += 1
        contributors = sorted(u[0] for u in units if u[3] > 0)
        assert contributors == list(range(oc + 1, q_end))
        for c, i, n, k0, k1 in units:
            if k0 > 0:
                assert i == dp_units[c], "a contributor unit must be its cluster's first stream-K unit"
                assert c < plan["sk_pairs"]


SHAPES = [(8192, 8192, 8192, 0), (4096, 4096, 4096, 0), (2048, 2048, 32768, 1), (6000, 5000, 3000, 0),
          (4096, 256, 65536, 0), (20480, 20480, 1024, 0), (600, 520, 776, 0)]


@pytest.mark.parametrize("M,N,K,dt", SHAPES)
@pytest.mark.parametrize("mode", [0, 2])
def test_stream_k_schedule(M, N, K, dt, mode):
    try:
        tc.gemm_f16_set_config(cta_group=2, stream_k=mode)
        for sms in (152, 148, 132):
            plan = tc.gemm_f16_plan(M, N, K, dt, num_sms=sms, with_workspace=True)
            check_plan(plan)
            if plan["sk_tiles"]:
                flags = -(-plan["sk_pairs"] * 8 * 4 // 256) * 256
                assert plan["workspace_bytes"] == flags + plan["sk_pairs"] * 2 * 128 * 256 * 4
    finally:
        tc.gemm_f16_set_config()


def test_planner_uses_stream_k_where_the_last_wave_is_thin():
    # 36 tail tiles of 1024, two equal K halves each, on 72 of the 76 pairs
    p = tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152, with_workspace=True)
    assert (p["dp_tiles"], p["sk_tiles"], p["sk_pairs"], p["grid"]) == (988, 36, 72, 152)
    p = tc.gemm_f16_plan(4096, 4096, 4096, 0, num_sms=152, with_workspace=True)
    assert (p["dp_tiles"], p["sk_tiles"], p["sk_pairs"]) == (228, 28, 56)
    # equal parts: pairs holding part j of different tail tiles run the same K range
    KB = p["k_steps"]
    S = p["sk_tiles"] * KB
    for c in range(p["sk_pairs"]):
        assert S * c // p["sk_pairs"] % KB == (c % 2) * KB // 2
    # 64 tiles on 76 pairs cannot be split evenly: data-parallel
    p = tc.gemm_f16_plan(2048, 2048, 32768, 1, num_sms=152, with_workspace=True)
    assert (p["dp_tiles"], p["sk_tiles"], p["grid"]) == (64, 0, 128)
    # 24 pair tiles on 76 pairs: three parts each on 72 pairs
    try:
        tc.gemm_f16_set_config(cta_group=2)
        p = tc.gemm_f16_plan(2048, 768, 8192, 0, num_sms=152, with_workspace=True)
        assert (p["num_tiles"], p["dp_tiles"], p["sk_tiles"], p["sk_pairs"], p["grid"]) == (24, 0, 24, 72, 144)
    finally:
        tc.gemm_f16_set_config()
    # a full last wave needs no stream-K: 76 x 2 tiles
    assert tc.gemm_f16_plan(256 * 38, 256 * 4, 4096, 0, num_sms=152, with_workspace=True)["sk_tiles"] == 0
    # tiny problems stay data-parallel (fewer than 8 iterations per sharing pair)
    assert tc.gemm_f16_plan(600, 520, 776, 0, num_sms=152, with_workspace=True)["sk_tiles"] == 0
    try:
        tc.gemm_f16_set_config(stream_k=1)
        assert tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152, with_workspace=True)["sk_tiles"] == 0
        with pytest.raises(tc.GemmError):
            tc.gemm_f16_set_config(stream_k=3)
    finally:
        tc.gemm_f16_set_config()
    p = tc.gemm_f16_plan(8192, 8192, 8192, 0, num_sms=152, with_workspace=True)
    assert tc.gemm_f16_workspace_size(8192, 8192, 8192, 0, num_sms=152) == p["workspace_bytes"] > 0
    assert tc.gemm_f16_workspace_size(600, 520, 776, 0, num_sms=152) == 0
