// The fp16 GEMM on a CTA pair (cta_group::2): a cluster of two CTAs on two
// SMs owns each PM x PN output tile, 256 x 256 for large problems and
// 128 x 128 for small ones.
//
// Same method as gemm_kernel.cuh (parallel grid of tiles, K pipeline through
// an mbarrier-guarded shared-memory ring, fp32 accumulator in TMEM, drain
// through shared memory and TMA; "Quickstart: GPU", section "Pipelining: a
// matmul kernel"), with the tile split over two SMs:
//   - CTA r (r = rank in the cluster) loads A rows [PM mb + PM/2 r, +PM/2)
//     and B columns [PN nb + PN/2 r, +PN/2) of each K step (256 x 256: 32 KiB
//     per 64-deep step each, where a 128 x 256 tile on one SM needs 48 KiB);
//   - one thread of the even CTA issues tcgen05.mma.cta_group::2 with M = PM,
//     N = PN: each SM's tensor core takes its PM/2 rows of A from its own
//     shared memory and the two halves of B from both, and writes its PM/2
//     rows of D into its own TMEM.  With M = 256 a CTA's 128 rows sit in the
//     128 TMEM lanes, all PN columns across.  With M = 128 its 64 rows are
//     folded over the lanes: lanes 0-63 hold columns 0 .. PN/2-1 of rows
//     0-63, lanes 64-127 columns PN/2 .. PN-1 of the same rows, in PN/2 TMEM
//     columns; so all four lane quadrants stay busy, and no partial sums
//     change hands as they do under split-K;
//   - both CTAs' loads count on the even CTA's `full` barrier (the leader arms
//     it for both); the MMA commits release the slot in both CTAs and signal
//     both epilogues (multicast); both CTAs' epilogue warps hand the
//     accumulator back on the even CTA's `tmem_empty` barrier;
//   - each CTA's epilogue drains its own PM/2 x PN block as the single-CTA
//     kernel does: epilogue warp q reads TMEM lanes 32q .. 32q+31, which hold
//     rows 32q .. of the block (M = 256), or rows 32 (q % 2) .. and columns
//     PN/2 (q / 2) .. (M = 128).
// Persistent: cluster c walks pair tiles c, c + clusters, ... in the grouped
// raster.  Programmatic dependent launch as in the single-CTA kernel: the
// producer waits for the previous kernel just before its first TMA load, the
// epilogue just before its first access to C or the workspace (after its dry
// drain, when it runs one), the MMA warp never.
//
// Stream-K (sk_tiles > 0): the K iterations of the tiles beyond the full
// waves are split evenly over the first sk_pairs clusters, which run their
// shares before their data-parallel tiles, so every cluster ends at about the
// same time.  A share that starts inside a tile is a contributor: it parks
// its fp32 partial (each CTA its 128 rows) in the workspace slot of this
// cluster, then each epilogue warp releases its flag.  A unit that starts a
// tile but does not finish it is the tile's owner: its epilogue waits
// (bounded) for the flags of the following clusters that hold the rest of the
// tile and adds their partials in cluster order before storing, while the
// cluster's MMAs go on with its next tile.  When the owner unit is its
// cluster's last (no data-parallel tiles), its epilogue warps instead sum the
// partials into the spare TMEM accumulator while the owner's own MMAs run.
// Owners only wait on contributors and contributors wait on nobody, so there
// is no cycle; all clusters are resident at once (the grid is capped at the
// clusters the GPU can hold).
#pragma once

#include "gemm_common.cuh"

namespace tcgemm {

constexpr int kPairBM = 256;  // tile rows per pair (MMA M) of the large-problem variant
constexpr int kPairBN = 256;  // tile columns per pair (MMA N) of the large-problem variant
static_assert(kPartialFloats == kBM * kPairBN, "one CTA's partial of a pair tile");

// SK: K depth of one pipeline step, 64 or 128.  A deeper step issues twice
// the MMAs per barrier wait and per commit, with the same bytes in flight.
// PM x PN: the pair's tile, 256 x 256 or 128 x 128.
template <int OUT, int SK = kBK, int PM = kPairBM, int PN = kPairBN>
struct PairLayout {
    static_assert(SK == 64 || SK == 128, "step K");
    static_assert((PM == 256 && PN == 256) || (PM == 128 && PN == 128), "pair tile");
    static constexpr int kRows = PM / 2;                     // rows of A and D per CTA
    static constexpr int kAtomBytes = kRows * 64 * 2;        // kRows rows x one 128-byte swizzle row
    static constexpr int kABytes = kRows * SK * 2;           // this CTA's rows: SK/64 atoms
    static constexpr int kBBoxBytes = SK * 64 * 2;           // 64 columns x SK rows of B
    static constexpr int kBBoxes = PN / 2 / 64;              // this CTA's PN/2 columns of B
    static constexpr int kBBytes = kBBoxes * kBBoxBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kOutCols = OUT == 0 ? 64 : 32;
    static constexpr int kStagingBytes = 32 * 128;
    static constexpr int kAccCols = PM == 256 ? PN : PN / 2;  // TMEM columns of one accumulator
    static_assert(kAccCols % 64 == 0, "partials move two 32-column chunks at a time");
    static constexpr int kTmemCols = 2 * kAccCols;            // two accumulators (256 x 256: all 512)
    // full[8], empty[8], tmem_full[2], tmem_empty[2], drain, dry
    static constexpr int kNumBars = 2 * kMaxStages + 6;
    static constexpr int kFixedBytes = 4 * 2 * kStagingBytes + kNumBars * 8 + 16;
    static constexpr int smem_bytes(int slots) { return slots * kStageBytes + kFixedBytes + 1024; }
};

// PF: the instance for small launches (one unit per pair, at most half the SMs),
// whose CTAs mostly start while the previous kernel in the stream still runs:
// each producer prefetches its own unit's first pf_steps K steps into L2
// before the dependency wait, so its loads after the wait hit L2.  (L2 is
// where the previous kernel's writes land, so a prefetched line is never
// stale.)  A separate instance: the extra code measurably slows the launches
// of the other instances even when it does not run.
template <int OUT, int SK, int PM = kPairBM, int PN = kPairBN, bool PF = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const KernelParams p) {
    using L = PairLayout<OUT, SK, PM, PN>;
    constexpr int kCols = L::kOutCols;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int S = p.slots;
    const Carve cv = carve(S, L::kABytes, L::kBBytes, L::kStagingBytes, L::kNumBars);
    const uint32_t sA = base + cv.a;
    const uint32_t sB = base + cv.b;
    const uint32_t sC = base + cv.c;
    const uint32_t bar0 = base + cv.bar;
#ifdef TCGEMM_CHECK
    // the carve-up fits the shared memory this launch has, checked before any
    // of it is written (both CTAs of every pair decide alike)
    if ((base - raw) + cv.end > ptx::dynamic_smem_size()) {
        if (threadIdx.x == 0) record_timeout(kSiteSmemBounds);
        return;
    }
#endif
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + cv.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + cv.misc + 4);
    // the parts of the carve-up, for the bounds-check build's tests
    const uint32_t ring_a = (uint32_t)S * L::kABytes, ring_b = (uint32_t)S * L::kBBytes;
    const uint32_t staging_all = 4u * 2u * L::kStagingBytes, bars = (uint32_t)L::kNumBars * 8u;
    (void)ring_a, (void)ring_b, (void)staging_all, (void)bars;

    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kMaxStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kMaxStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 4);
    const uint32_t dry_bar = bar0 + 8u * (2 * kMaxStages + 5);  // takes the dry drain's hand-back; never waited on

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Tracer tr(p, warp);  // warp w records as role w (trace build only)
    if (lane == 0) tr(kTrEntry, ptx::smid());
    const uint32_t rank = ptx::cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);   // the leader's arrive; both CTAs' bytes
            ptx::mbar_init(empty_bar(s), 1);  // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull_bar(a), 1);   // the leader's multicast commit
            ptx::mbar_init(tempty_bar(a), 8);  // 4 epilogue warps in each CTA
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(dry_bar, 8);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr((const void*)tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other (a
    // relaxed arrival: fence.mbarrier_init above released the initialisation)
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (lane == 0) tr(kTrSetup);

    const int cluster = blockIdx.x >> 1;   // this pair
    const int clusters = gridDim.x >> 1;
    const int KB = p.k_blocks;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0 && KB > 0 && p.inject == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            bool dep_done = false;
            UnitIter u;
            unit_iter_init(u, p, cluster, clusters);
            int t, k0, k1;
            if constexpr (PF) {
                UnitIter u2 = u;
                if (unit_next(u2, p, t, k0, k1)) {
                    int mb, nb;
                    tile_coords(t, p, mb, nb);
                    const int m0 = mb * PM + (int)rank * L::kRows;
                    const int n0 = nb * PN + (int)rank * (PN / 2);
                    const int kend = min(k1, k0 + p.pf_steps);
                    for (int kb = k0; kb < kend; ++kb) {
#pragma unroll
                        for (int h = 0; h < SK / 64; ++h) ptx::tma_prefetch_2d(&tmA, kb * SK + h * 64, m0);
#pragma unroll
                        for (int j = 0; j < L::kBBoxes; ++j) ptx::tma_prefetch_2d(&tmB, n0 + j * 64, kb * SK);
                    }
                }
            }
            while (ok && unit_next(u, p, t, k0, k1)) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int m0 = mb * PM + (int)rank * L::kRows;
                const int n0 = nb * PN + (int)rank * (PN / 2);
                // every second data-parallel tile walks K backwards: it starts on the
                // K range the cluster's previous tile (same row block of A) ended on,
                // still in L2
                const bool rev = k0 == 0 && k1 == KB && (u.ndp & 1) == 0;
                for (int kb0 = k0; kb0 < k1; ++kb0) {
                    const int kb = rev ? k1 - 1 - (kb0 - k0) : kb0;
                    if (!TC_CHECK(holds(bar0, bars, empty_bar(stage), 8) && holds(bar0, bars, full_bar(stage), 8) &&
                                      holds(sA, ring_a, sA + stage * L::kABytes, L::kABytes) &&
                                      holds(sB, ring_b, sB + stage * L::kBBytes, L::kBBytes),
                                  kSiteSmemBounds)) {
                        ok = false;
                        break;
                    }
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = full_bar(stage);
                    if (rank == 0) ptx::mbar_arrive_expect_tx(fb_local, 2 * L::kStageBytes);
                    const uint32_t fb = ptx::mapa(fb_local, 0);
                    if (!dep_done) {
                        // the previous kernel's writes of A and B are done from here on
                        ptx::grid_dependency_wait();
                        ptx::grid_launch_dependents();
                        tr(kTrDepWait);
                        dep_done = true;
                    }
#pragma unroll
                    for (int h = 0; h < SK / 64; ++h)
                        ptx::tma_load_2d_pair(sA + stage * L::kABytes + h * L::kAtomBytes, &tmA, fb, kb * SK + h * 64,
                                              m0);
#pragma unroll
                    for (int j = 0; j < L::kBBoxes; ++j)
                        ptx::tma_load_2d_pair(sB + stage * L::kBBytes + j * L::kBBoxBytes, &tmB, fb, n0 + j * 64,
                                              kb * SK);
                    tr(kTrLoad, kb);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the leader's full barriers count both CTAs' bytes: let every armed
            // phase land before shared memory goes away
            if (rank == 0)
                for (int s = 0; s < S; ++s)
                    if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_phase >> s) & 1u, p.wait_limit);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader only) ----------------
        if (lane == 0 && rank == 0 && KB > 0) {
            constexpr uint32_t idesc = make_idesc(PM, PN);
            int stage = 0;
            uint32_t phase = 0;
            long long it = 0;
            int tl = 0;
            bool ok = true;
            UnitIter u;
            unit_iter_init(u, p, cluster, clusters);
            int t, k0, k1;
            while (ok && unit_next(u, p, t, k0, k1)) {
                const int acc = tl & 1;
                const uint32_t aph = (tl >> 1) & 1;
                ++tl;
                if (!wait_bounded<true>(tempty_bar(acc), aph ^ 1u, abort_flag, p.wait_limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (!TC_CHECK((uint32_t)(acc * L::kAccCols + L::kAccCols) <= (uint32_t)L::kTmemCols, kSiteTmemBounds)) {
                    ok = false;
                    break;
                }
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * L::kAccCols);
                for (int kb = k0; kb < k1; ++kb) {
                    int rs = stage - p.release;
                    if (rs < 0) rs += S;
                    if (!TC_CHECK(holds(bar0, bars, full_bar(stage), 8) && holds(bar0, bars, empty_bar(rs), 8) &&
                                      holds(sA, ring_a, sA + stage * L::kABytes, L::kABytes) &&
                                      holds(sB, ring_b, sB + stage * L::kBBytes, L::kBBytes),
                                  kSiteSmemBounds)) {
                        ok = false;
                        break;
                    }
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, p.wait_limit, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    tr(kTrFull, kb);
                    const uint32_t a0 = sA + stage * L::kABytes;
                    const uint32_t b0 = sB + stage * L::kBBytes;
                    // descriptors of the step's first K slice; later slices add to
                    // the start-address field (16-byte units, no carry out of it)
                    const uint64_t ad0 = sw128_desc(a0, 16, 1024);
                    const uint64_t bd0 = sw128_desc(b0, L::kBBoxBytes, 1024);
#pragma unroll
                    for (int k = 0; k < SK / kUmmaK; ++k) {
                        // A K-major: slice k is 32 bytes along the swizzled row of atom k/4.
                        // B MN-major: slice k is two 8-row groups (2 KiB) further down;
                        // the 64-wide column blocks are one box apart.
                        const uint64_t ad = ad0 + (uint64_t)(((k / 4) * L::kAtomBytes + (k % 4) * (kUmmaK * 2)) >> 4);
                        const uint64_t bd = bd0 + (uint64_t)((k * (kUmmaK * 128)) >> 4);
                        ptx::mma_f16_ss_pair(d_tmem, ad, bd, idesc, (kb != k0) || (k != 0));
                    }
                    if (it >= p.release) ptx::mma_commit_pair_multicast(empty_bar(rs), 0x3);
                    ++it;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair_multicast(tfull_bar(acc), 0x3);
                tr(kTrTileDone, t);
            }
            ptx::mma_commit_pair(drain_bar);
            wait_drain(drain_bar, 0, p.wait_limit);
        }
    } else {
        // ---------------- epilogue (both CTAs): own PM/2 rows x PN columns ----------------
        const int q = warp & 3;
        const uint32_t staging = sC + (uint32_t)(q * 2 * L::kStagingBytes);
        const int row_in_tile = q * 32 + lane;  // TMEM lane: the workspace's row index
        // this warp's block of the CTA's PM/2 x PN: rows wrow .., columns wcol ..
        const int wrow = PM == 256 ? q * 32 : (q & 1) * 32;
        const int wcol = PM == 256 ? 0 : (q >> 1) * (PN / 2);
        int tl = 0;
        int nstore = 0;
        // every pair holds at most one tile, with no stream-K units
        const bool one_unit = p.sk_tiles == 0 && p.dp_tiles <= clusters;
        // the dry pass (below) touches no byte of global memory, so it runs
        // before the wait for the previous kernel; everything else after it
        const bool dry_first = one_unit && KB > 0;
        if (!dry_first) {
            // the previous kernel's reads and writes of C and of the workspace
            // are done from here on
            ptx::grid_dependency_wait();
            ptx::grid_launch_dependents();
            if (lane == 0) tr(kTrDepWait);
        }
        UnitIter u;
        unit_iter_init(u, p, cluster, clusters);
        int t, k0, k1;
        while (unit_next(u, p, t, k0, k1)) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int acc = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            ++tl;
            // stream-K owner (a unit that starts a tile without finishing it): the
            // workspace slots [s_first, s_end) hold the rest of the tile's K range
            int s_first = 0, s_end = 0;
            if (k0 == 0 && k1 < KB) sk_owner_slots(p, cluster, t, s_first, s_end);
            // bounds-check build: everything this unit's drain touches (this warp's
            // staging, both accumulators' columns, the workspace slots and flags)
            if (!(TC_CHECK(holds(sC, staging_all, staging, 2 * L::kStagingBytes), kSiteSmemBounds) &&
                  TC_CHECK(2u * L::kAccCols <= (uint32_t)L::kTmemCols, kSiteTmemBounds) &&
                  TC_CHECK(!(k0 > 0 || k1 < KB) ||
                               (2 * sk_slots(p) <= kMaxSkCtas && s_end <= sk_slots(p) &&
                                (k0 == 0 || sk_park_slot(p, cluster, t) < sk_slots(p))),
                           kSiteWorkspaceBounds)))
                break;
            const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
            // the cluster's last unit: once its accumulator is complete, every MMA
            // and load of this CTA is done and the operand ring is idle, so a drain
            // of more chunks than the two staging buffers hold stages every chunk
            // in a ring buffer of its own and issues the stores back to back; and
            // no MMA waits for the accumulator any more, so it is not handed back
            constexpr int kChunksPerWarp = L::kAccCols / kCols;
            bool last_unit = false, ring_drain = false;
            {
                UnitIter peek = u;
                int t2, a2, b2;
                last_unit = !unit_next(peek, p, t2, a2, b2);
                ring_drain = kChunksPerWarp > 2 && last_unit && KB > 0 && k0 == 0 &&
                             4u * kChunksPerWarp * 4096u <= ring_a + ring_b &&
                             TC_CHECK(holds(sA, ring_a + ring_b, sA + (uint32_t)(q * kChunksPerWarp * 4096),
                                            kChunksPerWarp * 4096u),
                                      kSiteSmemBounds);
            }
            bool prefetched = false;
            if (k0 == 0 && k1 < KB) {
                bool ok = true;
                for (int qq = s_first; ok && qq < s_end; ++qq) {
                    const unsigned* f = p.flags + (qq * 2 + (int)rank) * 4 + q;
                    int r = 1;
                    if (lane == 0) r = wait_flag(f, p.epoch, abort_flag, 4 * p.wait_limit);
                    ok = __shfl_sync(0xffffffffu, r, 0) != 0;
                    if (ok) (void)ptx::ld_acquire_gpu(f);  // orders this lane's reads after the flag
                }
                if (!ok) break;
                // every lane has acquired them: hand the flags back (zero), so a later
                // launch with the same epoch (a replayed CUDA graph) waits afresh
                __syncwarp();
                if (lane == 0) {
                    for (int qq = s_first; qq < s_end; ++qq) ptx::st_relaxed_gpu(p.flags + (qq * 2 + (int)rank) * 4 + q, 0u);
                    tr(kTrFlags, t);
                }
                // the owner unit is its cluster's last, so the other accumulator is
                // free: sum the contributors' partials into it while the MMAs run
                if (s_end > s_first && last_unit) {
                    const uint32_t spare = lane_base + (uint32_t)((acc ^ 1) * L::kAccCols);
                    // two 32-column chunks a round trip: the loads are latency-bound
#pragma unroll 1
                    for (int c = 0; c < L::kAccCols / 32; c += 2) {
                        uint32_t x0[32], x1[32];
                        for (int qq = s_first; qq < s_end; ++qq) {
                            const float* slot = p.ws + (size_t)(qq * 2 + (int)rank) * kPartialFloats;
                            uint32_t y0[32], y1[32];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                ptx::ld_global_cg_v4(slot + (size_t)(((c * 8 + j) * kBM + row_in_tile) * 4), y0[4 * j],
                                                     y0[4 * j + 1], y0[4 * j + 2], y0[4 * j + 3]);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                ptx::ld_global_cg_v4(slot + (size_t)((((c + 1) * 8 + j) * kBM + row_in_tile) * 4),
                                                     y1[4 * j], y1[4 * j + 1], y1[4 * j + 2], y1[4 * j + 3]);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                if (qq == s_first) {
                                    x0[i] = y0[i];
                                    x1[i] = y1[i];
                                } else {
                                    fadd_bits(x0[i], y0[i]);
                                    fadd_bits(x1[i], y1[i]);
                                }
                            }
                        }
                        ptx::tmem_st_32x32b_x32(spare + (uint32_t)(c * 32), x0);
                        ptx::tmem_st_32x32b_x32(spare + (uint32_t)((c + 1) * 32), x1);
                    }
                    ptx::tmem_st_wait();
                    prefetched = true;
                }
            }
            const int row0 = mb * PM + (int)rank * L::kRows + wrow;
            const int col0 = nb * PN + wcol;
            // A pair with a single tile (small problems) first runs the drain
            // once dry, before the wait for the previous kernel and while its
            // main loop runs: from the spare accumulator (never written then),
            // into this warp's staging, storing to rows from M on (clipped: no
            // byte written), handing back on a barrier nobody waits on.  The real
            // pass, on the critical path, then finds every instruction of it in
            // the instruction cache: the first run of each stretch of code
            // otherwise misses, ~500 cycles a time.
            bool failed = false;
#pragma unroll 1
            for (int pass = (dry_first && tl == 1) ? 0 : 1; pass < 2; ++pass) {
                const bool dry = pass == 0;
                if (dry_first && !dry) {
                    // the previous kernel's reads and writes of C are done from here on
                    ptx::grid_dependency_wait();
                    ptx::grid_launch_dependents();
                    if (lane == 0) tr(kTrDepWait);
                }
                if (KB > 0 && !dry) {
                    if (!warp_wait(tfull_bar(acc), aph, abort_flag, 4 * p.wait_limit, kSiteEpilogueTmemFull,
                                   lane)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (lane == 0) tr(kTrAccReady, t);
                }
                if (!dry && k0 > 0) break;  // stream-K contributor: parks its partial below
                const uint32_t trow = lane_base + (uint32_t)((dry ? acc ^ 1 : acc) * L::kAccCols);
#pragma unroll 1
                for (int c = 0; c < L::kAccCols / kCols; ++c) {
                    uint32_t v[kCols];
                    if (KB > 0) {
                        ptx::tmem_ld_32x32b_x32(trow + c * kCols, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                        if constexpr (OUT == 0)
                            ptx::tmem_ld_32x32b_x32(trow + c * kCols + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                        ptx::tmem_ld_wait();
                        if (c == L::kAccCols / kCols - 1) {
                            // this CTA's half of the accumulator is read: tell the leader
                            // (a release at cluster scope, ~1,000 cycles: not after the
                            // cluster's last unit, which no MMA waits for)
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0 && (dry || !last_unit))
                                ptx::mbar_arrive_cluster(ptx::mapa(dry ? dry_bar : tempty_bar(acc), 0));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kCols; ++i) v[i] = 0u;  // empty sum (K = 0)
                    }
                    // stream-K owner: add the contributors' partials (summed in slot
                    // order), from the spare accumulator or straight from the workspace
                    if (prefetched) {
                        uint32_t x[kCols];
                        const uint32_t sp = lane_base + (uint32_t)((acc ^ 1) * L::kAccCols + c * kCols);
                        ptx::tmem_ld_32x32b_x32(sp, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
                        if constexpr (OUT == 0) ptx::tmem_ld_32x32b_x32(sp + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                    }
                    for (int qq = s_first; !prefetched && qq < s_end; ++qq) {
                        const float* slot = p.ws + (size_t)(qq * 2 + (int)rank) * kPartialFloats;
                        uint32_t x[kCols];
#pragma unroll
                        for (int j = 0; j < kCols / 4; ++j)
                            ptx::ld_global_cg_v4(slot + (size_t)(((c * (kCols / 4) + j) * kBM + row_in_tile) * 4),
                                                 x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
#pragma unroll
                        for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                    }
                    add_c_in<OUT>(v, p, dry ? p.M : row0 + lane, col0 + c * kCols);  // row M: nothing read
                    store_chunk<OUT>(v, &tmC, staging, nstore, lane, col0 + c * kCols, dry ? p.M : row0,
                                     dry && p.M > (1 << 30),
                                     ring_drain && !dry ? sA + (uint32_t)((q * kChunksPerWarp + c) * 4096) : 0u);
                    if (!dry && lane == 0) tr(kTrStored, c);
                    if (dry) {
                        // one chunk runs all of the loop's code; the staging is free again
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                        nstore = 0;
                        break;
                    }
                }
            }
            if (failed) break;
            if (k0 > 0) {
                const uint32_t trow = lane_base + (uint32_t)(acc * L::kAccCols);
                // stream-K contributor: park this CTA's partial in its workspace slot
                // (the cluster's, or the tile's under helpers) as [TMEM column / 4]
                // [TMEM lane] 16-byte groups (consecutive lanes, consecutive 16 bytes),
                // then release the flag
                const int park = sk_park_slot(p, cluster, t);
                float* slot = p.ws + (size_t)(park * 2 + (int)rank) * kPartialFloats;
                // two 32-column chunks a TMEM round trip
#pragma unroll 1
                for (int c = 0; c < L::kAccCols / 32; c += 2) {
                    uint32_t v0[32], v1[32];
                    ptx::tmem_ld_32x32b_x32(trow + c * 32, v0);
                    ptx::tmem_ld_32x32b_x32(trow + (c + 1) * 32, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::st_global_v4(slot + (size_t)(((c * 8 + j) * kBM + row_in_tile) * 4), v0[4 * j],
                                          v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::st_global_v4(slot + (size_t)((((c + 1) * 8 + j) * kBM + row_in_tile) * 4), v1[4 * j],
                                          v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
                }
                // the flag first (an owner may be waiting on it), then the accumulator
                // back to the leader, unless this is the cluster's last unit
                ptx::tc_fence_before();
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    ptx::st_release_gpu(p.flags + (park * 2 + (int)rank) * 4 + q, p.epoch);
                    tr(kTrParked, t);
                    if (!last_unit) ptx::mbar_arrive_cluster(ptx::mapa(tempty_bar(acc), 0));
                }
                continue;
            }
        }
        if (lane == 0) {
            ptx::bulk_wait_group_read<0>();
            tr(kTrStoreRead);
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still signal into it.  The
    // arrival is relaxed: the barrier only marks that each CTA is done; what
    // crosses between the CTAs went through mbarriers, and the leader's MMAs,
    // which write the peer's Tensor Memory, completed (drain_bar) before its
    // arrival, so the peer frees its columns only after them.
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait();
    if (lane == 0) tr(kTrExit);
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
}

}  // namespace tcgemm
