// Persistent, warp-specialised fp16 GEMM for sm_103a: C[M,N] = A[M,K] * B[K,N],
// fp32 accumulation in Tensor Memory, fp16 or fp32 output.
//
// Method ("Quickstart: GPU", section "Pipelining: a matmul kernel";
// "JAX Pallas Mosaic GPU 快速上手", section "深入emit_pipeline的关键参数";
// "JAX Pallas 软件流水线 Software Pipelining 完全指南", sections 3, 4 and 9.2):
//   - a parallel grid of output tiles, each owned by exactly one block
//     (here: a persistent CTA walks tile ids in a grouped raster order);
//   - a sequential pipeline along K whose GMEM->SMEM copies overlap the
//     tensor-core work through a multi-buffered shared-memory ring
//     (max_concurrent_steps -> `stages` loads in flight);
//   - a buffer is reused only once the MMAs reading it have finished
//     (tcgen05.commit onto the slot's `empty` barrier), plus an optional
//     delay of `release` more steps (delay_release); the ring therefore has
//     slots = stages + release buffers;
//   - the fp32 accumulator (plgpu.ACC) lives in TMEM; the first K step of a
//     tile overwrites it instead of adding (the zero-init rule of the
//     software-pipelining guide's reduction example, section 7.2);
//   - the drain converts the accumulator to the output type, stages it in
//     shared memory, fences it for the async proxy and TMA-stores it.
//
// Split-K (split > 1): a cluster of `split` CTAs owns one tile; CTA rank r
// runs its own contiguous share of the K steps into its own TMEM, and the
// partial sums meet through distributed shared memory.  The tile's output
// column chunks are dealt out round-robin (chunk c belongs to rank c % split);
// a rank's partial of a chunk it does not own travels as one contiguous block
// per epilogue warp ([column / 4][row] 16-byte groups) into a ring buffer.
//   split = 2 (push): once its MMAs are done, each rank stores its partial of
//     the other's chunks straight from TMEM through registers into the other
//     CTA (st.async, counted as bytes on the other's `red_data` barrier).  The
//     blocks land in the receiving warp's output staging buffers, idle until
//     that warp drains, so a rank pushes as soon as its own MMAs are done and
//     the transfer overlaps the other rank's last steps.  When a warp's blocks
//     outgrow its staging (128 x 256 tiles), they land in the other's ring
//     instead, once the other reports it idle (`red_ready`).
//   split > 2 (pull): each rank parks the chunks it does not own in its own
//     ring, arrives on the others' `red_ready`, and reads the other ranks'
//     blocks of its own chunks over distributed shared memory.
// An owner adds the other ranks' partials to its own in ascending rank order
// (deterministic) and drains the sum as above.  The cluster barrier runs two
// phases: at set-up (every rank's barriers initialised before any remote
// arrive; only the epilogue waits on it there) and at exit (arrived at as
// soon as a thread is done with the other CTAs, waited on just before
// leaving), which keeps every rank's shared memory and barriers alive while
// the others may still touch them.  The planner gives each cluster exactly one
// tile in this mode.
//
// Stream-K (split = 1, sk_tiles > 0): as in the CTA-pair kernel, the K
// iterations of the shared tiles are dealt out in equal contiguous shares to
// sk_pairs CTAs, so every SM streams about the same number of K steps.  A
// CTA's first unit may start inside a tile: it is a contributor and parks its
// fp32 partial in its workspace slot, then each epilogue warp releases its
// flag.  A unit that starts a tile without finishing it is the tile's owner;
// it is its CTA's last unit, waits (bounded) for the flags of the following
// CTAs that hold the rest of the tile, and adds their partials in CTA order
// before storing.  Owners wait only on contributors, which wait on nobody;
// the grid never exceeds the CTAs the GPU holds at once.
//
// Programmatic dependent launch: the prologue (barriers, TMEM, tensor-map
// prefetch) and the producer's set-up of its first load (tile walk, first ring
// slot, expect-tx) run before `griddepcontrol.wait`, so they overlap the tail
// of the previous kernel in the stream.  Each role waits just before its first
// global-memory access: the producer before its first TMA load, the epilogue
// before its first access to C or the workspace (after its dry drain, when it
// runs one); the MMA warp touches only shared and tensor memory and never
// waits.  The set-up is worth moving: the first pass through each
// code path misses the instruction cache, about 500 cycles a time, and on
// the critical path after the wait those misses cost ~0.85 us per launch.
//
// Roles (192 threads, one CTA per SM):
//   warp 0       TMA producer (one lane)
//   warp 1       MMA issuer (one lane); allocates/frees TMEM (whole warp)
//   warps 2..5   epilogue; warp w reads TMEM lanes 32*(w%4) .. +31
#pragma once

#include "gemm_common.cuh"

namespace tcgemm {

template <int BN, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const KernelParams p) {
    using L = Layout<BN, OUT>;
    constexpr int kCols = L::kOutCols;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must sit on 1024-byte boundaries
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
    // of it is written (every CTA of the launch decides alike, so none is left
    // waiting on another)
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
    const uint32_t red_ready_bar = bar0 + 8u * (2 * kMaxStages + 5);
    const uint32_t red_data_bar = bar0 + 8u * (2 * kMaxStages + 6);
    const uint32_t dry_bar = bar0 + 8u * (2 * kMaxStages + 7);  // takes the dry drain's hand-back; never waited on
    // split-K parking: chunk c, epilogue warp quadrant q -> one contiguous
    // block of kCols / 4 column groups x 32 rows x 16 bytes in the ring
    constexpr int kChunks = BN / kCols;
    constexpr uint32_t kWarpChunkBytes = kCols / 4 * 32 * 16;
    auto park_at = [&](int c, int qd) { return sA + park_offset(c, qd, kWarpChunkBytes); };
    // split 2: the blocks a warp receives (its share of at most ceil(chunks / 2)
    // chunks) fit its two staging buffers for tiles up to 128 columns
    constexpr bool kPushToStaging = (kChunks + 1) / 2 * kWarpChunkBytes <= 2 * L::kStagingBytes;
    auto push_slot = [&](int c, int qd) {  // where chunk c's block of warp qd lands in its owner
        return kPushToStaging ? sC + push_offset(c, qd, kWarpChunkBytes, L::kStagingBytes) : park_at(c, qd);
    };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Tracer tr(p, warp);  // warp w records as role w (trace build only)
    if (lane == 0) tr(kTrEntry, ptx::smid());
    const int split = p.split;
    const uint32_t rank = split > 1 ? ptx::cluster_ctarank() : 0u;
    // split-K: the chunks this rank owns
    const int owned = (int)rank < kChunks ? (kChunks - (int)rank + split - 1) / split : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull_bar(a), 1);
            ptx::mbar_init(tempty_bar(a), 4);  // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        // split-K: the 4 epilogue warps of every other rank arrive on red_ready;
        // red_data (split 2): this CTA's own expect-tx arrival plus the pushed bytes
        ptx::mbar_init(red_ready_bar, split > 1 ? 4 * (split - 1) : 1);
        ptx::mbar_init(red_data_bar, 1);
        ptx::mbar_init(dry_bar, 4);
        // split 2: armed now for every byte the partner will push here
        if (split == 2 && owned > 0) ptx::mbar_arrive_expect_tx(red_data_bar, (uint32_t)owned * 4u * kWarpChunkBytes);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr((const void*)tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // Every CTA of the cluster has its barriers initialised before any remote
    // arrive.  The arrival is relaxed (fence.mbarrier_init above released the
    // initialisation; a release here costs ~1,000 cycles on the way to the
    // first load).  Only the epilogue, which signals and writes the other CTAs,
    // waits now; the producer and the MMA issuer touch nothing but their own
    // CTA and wait just before their second arrival, at the end.
    if (split > 1) {
        ptx::cluster_arrive_relaxed();
        if (warp >= 2) ptx::cluster_wait();
    }
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (lane == 0) tr(kTrSetup);

    // this CTA's cluster (itself without split-K) and the clusters of the grid
    const int cl = blockIdx.x / split;
    const int clusters = gridDim.x / split;
    // split-K: this rank's share of every tile's K steps, and the chunks it owns
    const int kb_begin = (int)((long long)p.k_blocks * rank / split);
    const int kb_end = (int)((long long)p.k_blocks * (rank + 1) / split);
    const bool has_k = p.k_blocks > 0;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        // (with the test hook set, nothing is loaded: the MMA warp's first wait
        // must run out and the whole CTA must wind down through the abort path)
        if (lane == 0 && has_k && p.inject == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;  // per slot: ever issued, parity of last issue
            bool ok = true;
            bool dep_done = false;
            UnitIter u;
            unit_iter_init(u, p, cl, clusters);
            int t, k0, k1;
            while (ok && unit_next(u, p, t, k0, k1)) {
                if (split > 1) k0 = kb_begin, k1 = kb_end;
                int mb, nb;
                tile_coords(t, p, mb, nb);
                // every second data-parallel tile of a CTA walks K backwards: it
                // starts on the K range the CTA's previous tile ended on, still in L2
                const bool rev = split == 1 && k0 == 0 && k1 == p.k_blocks && (u.ndp & 1) == 0;
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
                    const uint32_t fb = full_bar(stage);
                    ptx::mbar_arrive_expect_tx(fb, L::kStageBytes);
                    if (!dep_done) {
                        // the previous kernel's writes of A and B are done from here on
                        ptx::grid_dependency_wait();
                        ptx::grid_launch_dependents();
                        tr(kTrDepWait);
                        dep_done = true;
                    }
                    ptx::tma_load_2d(sA + stage * L::kABytes, &tmA, fb, kb * kBK, mb * kBM);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        ptx::tma_load_2d(sB + stage * L::kBBytes + j * kBoxBytes, &tmB, fb, nb * BN + j * 64,
                                         kb * kBK);
                    tr(kTrLoad, kb);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every load this CTA issued lands before shared memory goes away
            // (immediate in a normal run: the MMA warp consumed them all)
            for (int s = 0; s < S; ++s)
                if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_phase >> s) & 1u, p.wait_limit);
        }
        // split-K: the producer never touches another CTA (the set-up phase of
        // the cluster barrier completed long ago)
        if (split > 1) {
            ptx::cluster_wait();
            ptx::cluster_arrive();
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && has_k) {
            constexpr uint32_t idesc = make_idesc(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            long long it = 0;
            int tl = 0;
            bool ok = true;
            UnitIter u;
            unit_iter_init(u, p, cl, clusters);
            int t, k0, k1;
            while (ok && unit_next(u, p, t, k0, k1)) {
                if (split > 1) k0 = kb_begin, k1 = kb_end;
                const int acc = tl & 1;
                const uint32_t aph = (tl >> 1) & 1;
                ++tl;
                if (!wait_bounded(tempty_bar(acc), aph ^ 1u, abort_flag, p.wait_limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (!TC_CHECK((uint32_t)(acc * BN + BN) <= (uint32_t)L::kTmemCols, kSiteTmemBounds)) {
                    ok = false;
                    break;
                }
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
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
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // A K-major: a K slice of 16 is 32 bytes along the swizzled row.
                        // B MN-major: a K slice of 16 is two 8-row groups of 1024 bytes;
                        // consecutive 64-wide N blocks are one 8 KiB box apart.
                        const uint64_t ad = sw128_desc(a0 + k * (kUmmaK * 2), 16, 1024);
                        const uint64_t bd = sw128_desc(b0 + k * (kUmmaK * 128), kBoxBytes, 1024);
                        ptx::mma_f16_ss(d_tmem, ad, bd, idesc, (kb != k0) || (k != 0));
                    }
                    // release the slot `release` steps back once these MMAs are done
                    if (it >= p.release) ptx::mma_commit(empty_bar(rs));
                    ++it;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull_bar(acc));
                tr(kTrTileDone, t);
            }
            // every MMA this thread issued completes before TMEM is freed
            ptx::mma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.wait_limit);
        }
        if (split > 1) {
            ptx::cluster_wait();
            ptx::cluster_arrive();
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> SMEM -> TMA store ----------------
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t staging = sC + (uint32_t)(q * 2 * L::kStagingBytes);
        const int row_in_tile = q * 32 + lane;
        int tl = 0;
        int nstore = 0;
        bool arrived = false;
        // The first pass through the code that drains an accumulator misses the
        // instruction cache, ~500 cycles a stretch, on the critical path of a
        // small problem.  So when every CTA (under split-K every cluster) holds
        // a single tile, the epilogue runs that code once dry, before the wait
        // for the previous kernel and while the main loop runs: on the other
        // accumulator, storing to rows from M on (clipped: no byte of C
        // written), handing back on a barrier nobody waits on, pushing nothing.
        // Under split-K over two ranks the dry pass writes this CTA's staging,
        // which the partner pushes into: each rank arrives on the other's
        // `red_ready` once its dry pass is done, and waits on its own before
        // pushing (long done by then).
        const bool dry_ok = has_k && ((split == 1 && p.sk_tiles == 0 && p.dp_tiles <= clusters) ||
                                      (split == 2 && kPushToStaging));
        if (!dry_ok) {
            // the previous kernel's reads and writes of C (and of the workspace)
            // are done from here on
            ptx::grid_dependency_wait();
            ptx::grid_launch_dependents();
            if (lane == 0) tr(kTrDepWait);
        }
        UnitIter u;
        unit_iter_init(u, p, cl, clusters);
        int t, k0, k1;
        while (unit_next(u, p, t, k0, k1)) {
            if (split > 1) k0 = kb_begin, k1 = kb_end;
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int acc = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            ++tl;
            // bounds-check build: everything this unit's drain touches (this warp's
            // staging, both accumulators' columns, the split-K blocks, the
            // workspace slot and flags)
            bool in_bounds = TC_CHECK(holds(sC, staging_all, staging, 2 * L::kStagingBytes), kSiteSmemBounds) &&
                             TC_CHECK(2u * BN <= (uint32_t)L::kTmemCols, kSiteTmemBounds);
            for (int c = 0; in_bounds && split == 2 && c < kChunks; ++c)
                in_bounds = TC_CHECK(kPushToStaging ? holds(sC, staging_all, push_slot(c, q), kWarpChunkBytes)
                                                    : holds(sA, ring_a + ring_b, push_slot(c, q), kWarpChunkBytes),
                                     kSiteSmemBounds);
            for (int c = 0; in_bounds && split > 2 && c < kChunks; ++c)
                in_bounds = TC_CHECK(holds(sA, ring_a + ring_b, park_at(c, q), kWarpChunkBytes), kSiteSmemBounds);
            if (in_bounds && split == 1 && p.sk_tiles > 0)
                in_bounds = TC_CHECK(sk_park_slot(p, cl, t) < sk_slots(p) && sk_slots(p) <= kMaxSkCtas,
                                     kSiteWorkspaceBounds);
            if (!in_bounds) break;
            // a CTA's last unit without split-K: once its accumulator is complete,
            // every MMA and load of this CTA is done and the ring is idle (split-K
            // keeps partials there), so a drain of more chunks than the two
            // staging buffers hold stages every chunk in a ring buffer of its own
            // and issues the stores back to back
            constexpr int kChunksPerWarp = BN / kCols;
            bool ring_drain = false;
            if (kChunksPerWarp > 2 && split == 1 && has_k) {
                UnitIter peek = u;
                int t2, a2, b2;
                ring_drain = !unit_next(peek, p, t2, a2, b2) && 4u * kChunksPerWarp * 4096u <= ring_a + ring_b &&
                             TC_CHECK(holds(sA, ring_a + ring_b, sA + (uint32_t)(q * kChunksPerWarp * 4096),
                                            kChunksPerWarp * 4096u),
                                      kSiteSmemBounds);
            }
            // Dry pass first (see dry_ok): everything the code below does once
            // the accumulator is ready, on the other accumulator, with no store,
            // no push and no hand-back; the real pass then finds the code in the
            // instruction cache.
            bool failed = false;
#pragma unroll 1
            for (int pass = (dry_ok && tl == 1) ? 0 : 1; pass < 2; ++pass) {
                const bool dry = pass == 0;
                if (dry_ok && !dry) {
                    // the previous kernel's reads and writes of C are done from here on
                    ptx::grid_dependency_wait();
                    ptx::grid_launch_dependents();
                    if (lane == 0) tr(kTrDepWait);
                }
                if (has_k && !dry) {
                    // a legitimate wait here spans a whole tile's main loop: allow 4x
                    if (!warp_wait(tfull_bar(acc), aph, abort_flag, 4 * p.wait_limit, kSiteEpilogueTmemFull, lane)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (lane == 0) tr(kTrAccReady, t);
                }
                const int row0 = mb * kBM + q * 32;
                // the dry pass reads the other accumulator, which a CTA holding one tile never writes
                const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((dry ? acc ^ 1 : acc) * BN);

                if (split == 2) {
                    const uint32_t peer = rank ^ 1u;
                    if constexpr (!kPushToStaging) {
                        // this CTA's MMAs are done, so its ring is idle: the partner may push
                        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(red_ready_bar, peer));
                        if (!warp_wait<true>(red_ready_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceReady, lane)) {
                            failed = true;
                            break;
                        }
                    } else if (!dry) {
                        // the partner's dry pass, which wrote its staging, is done
                        if (!warp_wait<true>(red_ready_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceReady, lane)) {
                            failed = true;
                            break;
                        }
                    }
                    // this warp's rows of the partner's chunks: TMEM -> registers -> the
                    // partner (consecutive lanes, consecutive 16 bytes)
#pragma unroll 1
                    for (int c = 0; c < kChunks; ++c) {
                        if (c % 2 == (int)rank) continue;
#pragma unroll 1
                        for (int h = 0; h < kCols / 32; ++h) {
                            uint32_t v[32];
                            ptx::tmem_ld_32x32b_x32(trow + c * kCols + h * 32, v);
                            ptx::tmem_ld_wait();
                            if (dry) continue;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                ptx::st_async_v4(ptx::mapa(push_slot(c, q) + (uint32_t)(((h * 8 + j) * 32 + lane) * 16), peer),
                                                 v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3],
                                                 ptx::mapa(red_data_bar, peer));
                        }
                    }
                    if (!dry && lane == 0) tr(kTrPushed);
                    // the partner's blocks are waited for in the chunk loop below, after
                    // this CTA's own chunk has come out of TMEM
                } else if (split > 2) {
                    // park the partial of every chunk another rank owns in this CTA's
                    // ring: this warp's 32 rows as [column / 4][row] 16-byte groups
#pragma unroll 1
                    for (int c = 0; c < kChunks; ++c) {
                        if (c % split == (int)rank) continue;
#pragma unroll 1
                        for (int h = 0; h < kCols / 32; ++h) {
                            uint32_t v[32];
                            ptx::tmem_ld_32x32b_x32(trow + c * kCols + h * 32, v);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                ptx::st_shared_v4(park_at(c, q) + (uint32_t)(((h * 8 + j) * 32 + lane) * 16), v[4 * j],
                                                  v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        for (int r = 0; r < split; ++r)
                            if (r != (int)rank) ptx::mbar_arrive_cluster(ptx::mapa(red_ready_bar, (uint32_t)r));
                        tr(kTrPushed);
                    }
                    if (!warp_wait<true>(red_ready_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceReady, lane)) {
                        failed = true;
                        break;
                    }
                    if (lane == 0) tr(kTrPartner);
                } else if (k0 > 0) {
                    // stream-K contributor: park this CTA's partial in its workspace
                    // slot as [column / 4][row] 16-byte groups (consecutive lanes,
                    // consecutive 16 bytes), then release this warp's flag
                    const int park = sk_park_slot(p, cl, t);
                    float* slot = p.ws + (size_t)park * kPartialFloats;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t v[32];
                        ptx::tmem_ld_32x32b_x32(trow + c * 32, v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            ptx::st_global_v4(slot + (size_t)(((c * 8 + j) * kBM + row_in_tile) * 4), v[4 * j],
                                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::st_release_gpu(p.flags + park * 4 + q, p.epoch);
                        tr(kTrParked, t);
                    }
                    continue;
                }
                // stream-K owner: the workspace slots [s_first, s_end) (the CTAs after
                // this one whose shares start inside this tile) hold the rest of its K range
                int s_first = 0, s_end = 0;
                if (split == 1 && k1 < p.k_blocks) {
                    sk_owner_slots(p, cl, t, s_first, s_end);
                    bool ok = TC_CHECK(s_end <= sk_slots(p), kSiteWorkspaceBounds);
                    for (int qq = s_first; ok && qq < s_end; ++qq) {
                        const unsigned* f = p.flags + qq * 4 + q;
                        int r = 1;
                        if (lane == 0) r = wait_flag(f, p.epoch, abort_flag, 4 * p.wait_limit);
                        ok = __shfl_sync(0xffffffffu, r, 0) != 0;
                        if (ok) (void)ptx::ld_acquire_gpu(f);  // orders this lane's reads after the flag
                    }
                    if (!ok) {
                        failed = true;
                        break;
                    }
                    // every lane has acquired them: hand the flags back (zero), so a later
                    // launch with the same epoch (a replayed CUDA graph) waits afresh
                    __syncwarp();
                    if (lane == 0) {
                        for (int qq = s_first; qq < s_end; ++qq) ptx::st_relaxed_gpu(p.flags + qq * 4 + q, 0u);
                        tr(kTrFlags, t);
                    }
                }

#pragma unroll 1
                for (int c = 0; c < BN / kCols; ++c) {
                    if (split > 1 && c % split != (int)rank) continue;
                    uint32_t v[kCols];
                    if (has_k) {
                        ptx::tmem_ld_32x32b_x32(trow + c * kCols, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                        if constexpr (OUT == 0)
                            ptx::tmem_ld_32x32b_x32(trow + c * kCols + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                        ptx::tmem_ld_wait();
                        if (split == 1 && c == BN / kCols - 1) {
                            // accumulator fully read: hand it back to the MMA warp
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(dry ? dry_bar : tempty_bar(acc));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kCols; ++i) v[i] = 0u;  // empty sum (K = 0)
                    }
                    if (split == 2) {
                        if (!dry && !arrived) {
                            // the partner's blocks of this CTA's chunks
                            if (!warp_wait<true>(red_data_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceData, lane)) {
                                failed = true;
                                break;
                            }
                            if (lane == 0) tr(kTrPartner);
                            // done with the partner: its pushes have landed here, and it arrives
                            // only once this CTA's pushes have landed there (the barrier keeps
                            // shared memory alive; the data went through mbarriers, so the
                            // arrival need not release anything)
                            ptx::cluster_arrive_relaxed();
                            arrived = true;
                        }
                        // the partner's partial, pushed into this CTA
                        uint32_t x[kCols];
#pragma unroll
                        for (int j = 0; j < kCols / 4; ++j)
                            ptx::ld_shared_v4(push_slot(c, q) + (uint32_t)((j * 32 + lane) * 16), x[4 * j], x[4 * j + 1],
                                              x[4 * j + 2], x[4 * j + 3]);
                        // every lane has its values before any lane reuses the staging
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                    } else if (split > 2) {
                        // add the other ranks' partials to this rank's own, in ascending
                        // rank order: a fixed order, so the result is deterministic
                        for (int r = 0; r < split; ++r) {
                            if (r == (int)rank) continue;
                            // all of the chunk's remote loads in flight at once, then the adds
                            uint32_t x[kCols];
#pragma unroll
                            for (int j = 0; j < kCols / 4; ++j)
                                ptx::ld_cluster_v4(ptx::mapa(park_at(c, q) + (uint32_t)((j * 32 + lane) * 16), (uint32_t)r),
                                                   x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
#pragma unroll
                            for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                        }
                    }
                    // stream-K owner: add the contributors' partials, in slot (CTA) order
                    for (int qq = s_first; qq < s_end; ++qq) {
                        const float* slot = p.ws + (size_t)qq * kPartialFloats;
                        uint32_t x[kCols];
#pragma unroll
                        for (int j = 0; j < kCols / 4; ++j)
                            ptx::ld_global_cg_v4(slot + (size_t)(((c * (kCols / 4) + j) * kBM + row_in_tile) * 4),
                                                 x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
#pragma unroll
                        for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                    }
                    add_c_in<OUT>(v, p, dry ? p.M : row0 + lane, nb * BN + c * kCols);  // row M: nothing read
                    store_chunk<OUT>(v, &tmC, staging, nstore, lane, nb * BN + c * kCols, dry ? p.M : row0,
                                     dry && p.M > (1 << 30),
                                     ring_drain && !dry ? sA + (uint32_t)((q * kChunksPerWarp + c) * 4096) : 0u);
                    if (!dry && lane == 0) tr(kTrStored, c);
                    if (dry) {
                        // one chunk runs all of the loop's code; the staging is free
                        // again and the real pass starts on buffer 0 (under split-K
                        // the partner's pushed partials sit in both buffers)
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                        nstore = 0;
                        break;
                    }
                }
                if (failed) break;
                // split-K over two ranks: this CTA's staging is the partner's to push into
                if (dry && split == 2) {
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(red_ready_bar, rank ^ 1u));
                }
            }
            if (failed) break;
        }
        // after an abort: bytes the partner may still push land before this CTA leaves
        if (split == 2 && owned > 0 && warp == 2 && lane == 0) wait_drain(red_data_bar, 0, p.wait_limit);
        // the staging buffers must have been read before shared memory goes
        // away; the global writes themselves complete with the grid
        if (lane == 0) {
            ptx::bulk_wait_group_read<0>();
            tr(kTrStoreRead);
        }
        __syncwarp();
        if (split > 1 && !arrived) ptx::cluster_arrive();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // split-K: no rank leaves while another may still read or write its
    // shared memory or arrive on its barriers
    if (split > 1) ptx::cluster_wait();
    if (lane == 0) tr(kTrExit);
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

}  // namespace tcgemm
