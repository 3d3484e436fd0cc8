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
// column chunks are dealt out round-robin (chunk c belongs to rank c % split).
// Every rank parks its fp32 partial of the chunks it does not own in its (now
// idle) ring buffers and arrives on the other ranks' `red_ready` barriers;
// each rank then adds, for the chunks it owns, the other ranks' partials to
// its own in ascending rank order (deterministic), drains them as above, and arrives on the others'
// `red_done`, which keeps every rank's shared memory alive until it is read.
// The planner gives each cluster exactly one tile in this mode.
//
// Programmatic dependent launch: the prologue (barriers, TMEM, tensor-map
// prefetch) runs before `griddepcontrol.wait`, so it overlaps the tail of the
// previous kernel in the stream; no global memory is touched before the wait.
//
// Roles (192 threads, one CTA per SM):
//   warp 0       TMA producer (one lane)
//   warp 1       MMA issuer (one lane); allocates/frees TMEM (whole warp)
//   warps 2..5   epilogue; warp w reads TMEM lanes 32*(w%4) .. +31
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace tcgemm {

constexpr int kBM = 128;       // tile rows = M of one cta_group::1 MMA = TMEM lanes
constexpr int kBK = 64;        // K per pipeline step: one 128-byte swizzle row of fp16
constexpr int kUmmaK = 16;     // K of one tcgen05.mma with 16-bit operands
constexpr int kThreads = 192;  // 6 warps
constexpr int kMaxStages = 8;
constexpr int kMaxSplit = 8;   // portable cluster size
constexpr int kBoxBytes = kBK * 64 * 2;  // one 64 x 64 fp16 box of B: 8 KiB

// Status word written by a CTA whose bounded wait ran out (first writer wins).
enum WaitSite : unsigned {
    kSiteNone = 0,
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteEpilogueTmemFull = 4,
    kSiteDrain = 5,
    kSiteReduceReady = 6,
    kSiteReduceDone = 7,
};

__device__ unsigned int g_status;

struct KernelParams {
    int M, N, K;
    int tiles_m, tiles_n, k_blocks;
    int raster_group;      // m-blocks per raster group
    int slots;             // ring buffers = stages in flight + release depth, 1 .. kMaxStages
    int release;           // extra release depth, 0 .. slots-1
    int split;             // CTAs (one cluster) sharing a tile along K; 1 = no split
    long long wait_limit;  // clock cycles a single wait may take before giving up
    int inject;            // test hook: 1 = the producer issues no loads at all
};

template <int BN, int OUT>
struct Layout {
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile N");
    static constexpr int kABytes = kBM * kBK * 2;  // 16 KiB
    static constexpr int kBBytes = kBK * BN * 2;   // BN/64 boxes of 8 KiB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kOutCols = OUT == 0 ? 64 : 32;  // columns in one 128-byte output row
    static constexpr int kStagingBytes = 32 * 128;       // one warp's 32 rows x 128 bytes
    static constexpr int kTmemCols = 2 * BN;             // two accumulators
    static constexpr int kPartialBytes = kBM * BN * 4;   // one fp32 partial tile (split-K)
    // full[8], empty[8], tmem_full[2], tmem_empty[2], drain, red_ready, red_done
    static constexpr int kNumBars = 2 * kMaxStages + 7;
    static constexpr int kFixedBytes = 4 * 2 * kStagingBytes + kNumBars * 8 + 16;
    static constexpr int smem_bytes(int slots) { return slots * kStageBytes + kFixedBytes + 1024; }
};

// Instruction descriptor, kind::f16: D fp32, A and B fp16, A K-major, B
// MN-major (B is [K,N] with N contiguous), M = 128, N = BN.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4)                            // D format: fp32
           | (0u << 7) | (0u << 10)             // A, B format: fp16
           | (0u << 15)                         // A: K-major
           | (1u << 16)                         // B: MN-major
           | ((uint32_t)(n >> 3) << 17)         // N / 8
           | ((uint32_t)(m >> 4) << 24);        // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
// lbo/sbo in bytes; version 1 (tcgen05); swizzle mode 2 = 128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Grouped raster: groups of `g` m-blocks; inside a group the m-block varies
// fastest, so consecutive tile ids share B columns and a few A rows in L2.
__device__ __forceinline__ void tile_coords(int t, const KernelParams& p, int& mb, int& nb) {
    const int g = p.raster_group;
    const int per_group = g * p.tiles_n;
    const int grp = t / per_group;
    const int first_m = grp * g;
    const int gm = min(p.tiles_m - first_m, g);
    const int r = t - grp * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

__device__ __forceinline__ void record_timeout(unsigned site) { atomicCAS(&g_status, 0u, site); }

// Bounded wait on an mbarrier phase.  Gives up (returning false) when the
// CTA-wide abort flag is raised or, after `limit` cycles, raises it itself.
// kClusterAcquire: acquire at cluster scope (the data was written by another
// CTA of the cluster before it arrived).
template <bool kClusterAcquire = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             long long limit, unsigned site) {
    auto probe = [&]() {
        return kClusterAcquire ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const long long t0 = clock64();
    while (!probe()) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            record_timeout(site);
            return false;
        }
    }
    return true;
}

// Bounded wait that ignores the abort flag: used after an abort to let the
// CTA's own asynchronous copies and MMAs land before it exits.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            record_timeout(kSiteDrain);
            return false;
        }
    }
    return true;
}

// Lane 0 waits, the warp follows its verdict.
template <bool kClusterAcquire = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, long long limit,
                                          unsigned site, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bounded<kClusterAcquire>(bar, parity, abort_flag, limit, site);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One 128-byte-wide column chunk of a warp's 32 output rows: convert, write
// to the warp's staging buffer in the 128-byte swizzle the C tensor map
// expects (16-byte chunk j of row `lane` at chunk j ^ (lane % 8)), fence for
// the async proxy and TMA-store it.  Staging is double-buffered per warp.
template <int OUT>
__device__ __forceinline__ void store_chunk(const uint32_t (&v)[OUT == 0 ? 64 : 32], const CUtensorMap* tmC,
                                            uint32_t staging, int& nstore, int lane, int x, int y) {
    const uint32_t stg = staging + (uint32_t)((nstore & 1) * 4096);
    // the store issued from this buffer two rounds ago must have read it
    if (lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row_addr = stg + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w0, w1, w2, w3;
        if constexpr (OUT == 0) {
            w0 = ptx::pack_f16x2(v[8 * j + 0], v[8 * j + 1]);
            w1 = ptx::pack_f16x2(v[8 * j + 2], v[8 * j + 3]);
            w2 = ptx::pack_f16x2(v[8 * j + 4], v[8 * j + 5]);
            w3 = ptx::pack_f16x2(v[8 * j + 6], v[8 * j + 7]);
        } else {
            w0 = v[4 * j + 0];
            w1 = v[4 * j + 1];
            w2 = v[4 * j + 2];
            w3 = v[4 * j + 3];
        }
        ptx::st_shared_v4(row_addr + ((uint32_t)(j ^ (lane & 7)) << 4), w0, w1, w2, w3);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_2d(tmC, stg, x, y);
        ptx::bulk_commit_group();
    }
    ++nstore;
}

__device__ __forceinline__ void fadd_bits(uint32_t& acc, uint32_t add) {
    acc = __float_as_uint(__uint_as_float(acc) + __uint_as_float(add));
}

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
    const uint32_t sA = base;
    const uint32_t sB = sA + S * L::kABytes;
    const uint32_t sC = sB + S * L::kBBytes;
    const uint32_t bar0 = sC + 4 * 2 * L::kStagingBytes;
    const uint32_t misc_off = (bar0 - base) + L::kNumBars * 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + misc_off + 4);

    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kMaxStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kMaxStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 4);
    const uint32_t red_ready_bar = bar0 + 8u * (2 * kMaxStages + 5);
    const uint32_t red_done_bar = bar0 + 8u * (2 * kMaxStages + 6);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = p.split;
    const uint32_t rank = split > 1 ? ptx::cluster_ctarank() : 0u;

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
        // split-K: the 4 epilogue warps of every other rank arrive on these
        ptx::mbar_init(red_ready_bar, split > 1 ? 4 * (split - 1) : 1);
        ptx::mbar_init(red_done_bar, split > 1 ? 4 * (split - 1) : 1);
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
    // every CTA of the cluster has its barriers initialised before any remote arrive
    if (split > 1) ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the previous kernel's writes (and reads) of A, B and C are done from here on
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const int num_tiles = p.tiles_m * p.tiles_n;
    const int first_tile = blockIdx.x / split;
    const int tile_stride = gridDim.x / split;
    // this CTA's share of the K steps (all of them without split-K)
    const int kb_begin = (int)((long long)p.k_blocks * rank / split);
    const int kb_end = (int)((long long)p.k_blocks * (rank + 1) / split);
    const int KB = kb_end - kb_begin;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        // (with the test hook set, nothing is loaded: the MMA warp's first wait
        // must run out and the whole CTA must wind down through the abort path)
        if (lane == 0 && KB > 0 && p.inject == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;  // per slot: ever issued, parity of last issue
            bool ok = true;
            for (int t = first_tile; ok && t < num_tiles; t += tile_stride) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    ptx::mbar_arrive_expect_tx(fb, L::kStageBytes);
                    ptx::tma_load_2d(sA + stage * L::kABytes, &tmA, fb, kb * kBK, mb * kBM);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        ptx::tma_load_2d(sB + stage * L::kBBytes + j * kBoxBytes, &tmB, fb, nb * BN + j * 64,
                                         kb * kBK);
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
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && KB > 0) {
            constexpr uint32_t idesc = make_idesc(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            long long it = 0;
            int tl = 0;
            bool ok = true;
            for (int t = first_tile; ok && t < num_tiles; t += tile_stride, ++tl) {
                const int acc = tl & 1;
                const uint32_t aph = (tl >> 1) & 1;
                if (!wait_bounded(tempty_bar(acc), aph ^ 1u, abort_flag, p.wait_limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, p.wait_limit, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = sA + stage * L::kABytes;
                    const uint32_t b0 = sB + stage * L::kBBytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // A K-major: a K slice of 16 is 32 bytes along the swizzled row.
                        // B MN-major: a K slice of 16 is two 8-row groups of 1024 bytes;
                        // consecutive 64-wide N blocks are one 8 KiB box apart.
                        const uint64_t ad = sw128_desc(a0 + k * (kUmmaK * 2), 16, 1024);
                        const uint64_t bd = sw128_desc(b0 + k * (kUmmaK * 128), kBoxBytes, 1024);
                        ptx::mma_f16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0);
                    }
                    // release the slot `release` steps back once these MMAs are done
                    if (it >= p.release) {
                        int rs = stage - p.release;
                        if (rs < 0) rs += S;
                        ptx::mma_commit(empty_bar(rs));
                    }
                    ++it;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull_bar(acc));
            }
            // every MMA this thread issued completes before TMEM is freed
            ptx::mma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.wait_limit);
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> SMEM -> TMA store ----------------
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t staging = sC + (uint32_t)(q * 2 * L::kStagingBytes);
        const int row_in_tile = q * 32 + lane;
        int tl = 0;
        int nstore = 0;
        for (int t = first_tile; t < num_tiles; t += tile_stride, ++tl) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const int acc = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            if (KB > 0) {
                // a legitimate wait here spans a whole tile's main loop: allow 4x
                if (!warp_wait(tfull_bar(acc), aph, abort_flag, 4 * p.wait_limit, kSiteEpilogueTmemFull, lane))
                    break;
                ptx::tc_fence_after();
            }
            const int row0 = mb * kBM + q * 32;
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);

            if (split > 1) {
                // park the partial of every chunk another rank owns, laid out as
                // [column / 4][row] 16-byte groups so consecutive lanes touch
                // consecutive 16 bytes (no bank conflicts, here or in the remote reads)
#pragma unroll 1
                for (int c = 0; c < BN / kCols; ++c) {
                    if (c % split == (int)rank) continue;
#pragma unroll 1
                    for (int h = 0; h < kCols / 32; ++h) {
                        uint32_t v[32];
                        const int col = c * kCols + h * 32;
                        if (KB > 0) {
                            ptx::tmem_ld_32x32b_x32(trow + col, v);
                            ptx::tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = 0u;
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            ptx::st_shared_v4(sA + (uint32_t)(((col / 4 + j) * kBM + row_in_tile) * 16), v[4 * j],
                                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    for (int r = 0; r < split; ++r)
                        if (r != (int)rank) ptx::mbar_arrive_cluster(ptx::mapa(red_ready_bar, (uint32_t)r));
                if (!warp_wait<true>(red_ready_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceReady, lane)) break;
            }

#pragma unroll 1
            for (int c = 0; c < BN / kCols; ++c) {
                if (split > 1 && c % split != (int)rank) continue;
                uint32_t v[kCols];
                if (KB > 0) {
                    ptx::tmem_ld_32x32b_x32(trow + c * kCols, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                    if constexpr (OUT == 0)
                        ptx::tmem_ld_32x32b_x32(trow + c * kCols + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                    ptx::tmem_ld_wait();
                    if (split == 1 && c == BN / kCols - 1) {
                        // accumulator fully read: hand it back to the MMA warp
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kCols; ++i) v[i] = 0u;  // empty sum (K = 0)
                }
                if (split > 1) {
                    // add the other ranks' partials to this rank's own, in ascending
                    // rank order: a fixed order, so the result is deterministic
                    for (int r = 0; r < split; ++r) {
                        if (r == (int)rank) continue;
                        // all of the chunk's remote loads in flight at once, then the adds
                        uint32_t x[kCols];
#pragma unroll
                        for (int j = 0; j < kCols / 4; ++j) {
                            const int g = c * (kCols / 4) + j;  // 16-byte column group
                            ptx::ld_cluster_v4(ptx::mapa(sA + (uint32_t)((g * kBM + row_in_tile) * 16), (uint32_t)r),
                                               x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
                        }
#pragma unroll
                        for (int i = 0; i < kCols; ++i) fadd_bits(v[i], x[i]);
                    }
                }
                store_chunk<OUT>(v, &tmC, staging, nstore, lane, nb * BN + c * kCols, row0);
            }
            if (split > 1) {
                // this rank has read every partial it needs; wait until the others
                // have read this rank's before its shared memory may go away
                __syncwarp();
                if (lane == 0)
                    for (int r = 0; r < split; ++r)
                        if (r != (int)rank) ptx::mbar_arrive_cluster(ptx::mapa(red_done_bar, (uint32_t)r));
                warp_wait(red_done_bar, 0, abort_flag, 4 * p.wait_limit, kSiteReduceDone, lane);
            }
        }
        // the staging buffers must have been read before shared memory goes
        // away; the global writes themselves complete with the grid
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

}  // namespace tcgemm
