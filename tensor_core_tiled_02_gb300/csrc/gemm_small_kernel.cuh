// Small problems: one CTA per NT x 64 output tile (NT = 8, 16 or 32 rows of
// C by 64 columns), every K step loaded at once, one wave of up to one CTA
// per SM.  A launch this small is latency: what counts is the bytes each SM
// must take in before its MMAs can run (an NT x 64 tile needs NT + 64 rows
// of K per SM, where a 128 x 128 pair tile needs 128) and the fixed path
// from the dependency wait to the last store.
//
// The tile is computed transposed, D = C^T = B^T A^T, so that the MMA's M is
// the 64 columns of C and its N is the NT rows: tcgen05.mma kind::f16 with
// M = 64 and N = NT.  Its A operand is B's [64 columns x K] block as TMA
// loads it (MN-major, 128-byte swizzle: K rows of 128 bytes), its B operand
// A's [NT rows x K] block (K-major, 128-byte swizzle), so both come straight
// from the row-major inputs.  With M = 64 the accumulator row n (a column of
// C) lives in TMEM lane 32 (n / 16) + n % 16 and column m (a row of C): each
// epilogue warp holds 16 columns of C in its lanes 0..15, transposes them
// through shared memory (fp32) and stores NT rows of 128 (fp16) or 256 (fp32)
// bytes with plain coalesced stores, clipped at M and N, adding C's values
// first for C += A B.
//
// Roles (128 threads): warp 0 lane 0 issues every TMA load, one mbarrier per
// 64-deep K block, right after the dependency wait; warp 1 allocates TMEM and
// its lane 0 issues 4 MMAs per K block as each lands, then commits; all four
// warps drain.  Every wait is bounded and reports through the status word.
#pragma once

#include "gemm_common.cuh"

namespace tcgemm {

constexpr int kSmallBN = 64;       // columns of C per CTA (the MMA's M)
constexpr int kSmallMaxKB = 8;     // K blocks of 64 a launch may hold (K <= 512)
constexpr int kSmallThreads = 128;

template <int OUT, int NT>
struct SmallLayout {
    static_assert(NT == 8 || NT == 16 || NT == 32, "rows of C per CTA");
    static constexpr int kBtBytes = kSmallBN * 64 * 2;   // B block: 64 K rows x 128 bytes
    static constexpr int kABytes = NT * 64 * 2;          // A block: NT rows x 128 bytes
    static constexpr int kBlockBytes = kBtBytes + (kABytes < 1024 ? 1024 : kABytes);  // 1 KiB aligned parts
    static constexpr int kOutBytes = OUT == 0 ? 2 : 4;
    static constexpr int kStageBytes = NT * kSmallBN * 4;  // the C tile in fp32, row-major
    static constexpr int kTmemCols = 32;
    static constexpr int smem_bytes(int kb) { return kb * kBlockBytes + kStageBytes + (kSmallMaxKB + 1) * 8 + 16 + 1024; }
};

template <int OUT, int NT>
__global__ void __launch_bounds__(kSmallThreads, 1)
    gemm_f16_small_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          void* __restrict__ C, const KernelParams p) {
    using L = SmallLayout<OUT, NT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int KB = p.k_blocks;
    const uint32_t blocks = base;                                     // KB x (B block, A block)
    const uint32_t stage = base + (uint32_t)(KB * L::kBlockBytes);    // the C tile
    const uint32_t bar0 = stage + (uint32_t)L::kStageBytes;           // full[KB], done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + (bar0 - base) + (kSmallMaxKB + 1) * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t done_bar = bar0 + 8u * kSmallMaxKB;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Tracer tr(p, warp);  // warp w records as role w (trace build only)
    if (lane == 0) tr(kTrEntry, ptx::smid());
    // this CTA's tile: 64 columns of C from n0, NT rows from m0
    const int n0 = (int)(blockIdx.x % (uint32_t)p.tiles_n) * kSmallBN;
    const int m0 = (int)(blockIdx.x / (uint32_t)p.tiles_n) * NT;
    // K fits the blocks (the planner's rule) and the carve-up fits this
    // launch's shared memory (checked in the bounds-check build)
    const bool fits = KB >= 1 && KB <= kSmallMaxKB &&
                      TC_CHECK(bar0 + 8u * (kSmallMaxKB + 1) + 8u <= raw + ptx::dynamic_smem_size(), kSiteSmemBounds);

    if (threadIdx.x == 0) {
        for (int b = 0; b <= kSmallMaxKB; ++b) ptx::mbar_init(bar0 + 8u * b, 1);
        *abort_flag = fits ? 0 : 1;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr((const void*)tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool go = *abort_flag == 0;
    if (lane == 0) tr(kTrSetup);

    if (warp == 0) {
        // ---------------- TMA producer: every block at once ----------------
        // (with the test hook set nothing is loaded: the MMA warp's first wait
        // must run out and the CTA wind down through the abort path)
        if (lane == 0 && go && p.inject == 0) {
            // the CTA mostly starts while the previous kernel in the stream still
            // runs: ask L2 for its operands first, so that the loads after the
            // wait hit L2 (where the previous kernel's writes land, so a
            // prefetched line is never stale)
            for (int kb = 0; kb < KB; ++kb) {
                ptx::tma_prefetch_2d(&tmB, n0, kb * 64);
                ptx::tma_prefetch_2d(&tmA, kb * 64, m0);
            }
            // the previous kernel's writes of A and B are done from here on
            ptx::grid_dependency_wait();
            ptx::grid_launch_dependents();
            tr(kTrDepWait);
            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t fb = bar0 + 8u * kb;
                const uint32_t bt = blocks + (uint32_t)(kb * L::kBlockBytes);
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)(L::kBtBytes + L::kABytes));
                ptx::tma_load_2d(bt, &tmB, fb, n0, kb * 64);
                ptx::tma_load_2d(bt + L::kBtBytes, &tmA, fb, kb * 64, m0);
                tr(kTrLoad, kb);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && go) {
            // D (64 x NT, fp32) = B^T (MN-major) x A^T (K-major)
            constexpr uint32_t idesc = (1u << 4)                        // D fp32
                                       | (1u << 15)                     // A operand MN-major
                                       | ((uint32_t)(NT >> 3) << 17)    // N / 8
                                       | ((uint32_t)(kSmallBN >> 4) << 24);  // M / 16
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++kb) {
                ok = wait_bounded(bar0 + 8u * kb, 0, abort_flag, p.wait_limit, kSiteMmaFull);
                if (!ok) break;
                ptx::tc_fence_after();
                tr(kTrFull, kb);
                const uint32_t bt = blocks + (uint32_t)(kb * L::kBlockBytes);
                const uint64_t ad0 = sw128_desc(bt, L::kBtBytes, 1024);
                const uint64_t bd0 = sw128_desc(bt + L::kBtBytes, 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // K = 16 slice k: 16 rows (2 KiB) down the B block, 32 bytes along A's rows
                    const uint64_t ad = ad0 + (uint64_t)((k * 2048) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((k * 32) >> 4);
                    ptx::mma_f16_ss(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
            }
            // arrives once every MMA issued has completed (also after an abort,
            // so the drain below never leaves an MMA writing freed columns)
            ptx::mma_commit(done_bar);
            tr(kTrTileDone, blockIdx.x);
        }
    }

    // ---------------- epilogue: all four warps ----------------
    bool have = false;
    if (go) {
        ptx::grid_dependency_wait();  // the previous kernel's reads of C are done
        have = warp_wait(done_bar, 0, abort_flag, 4 * p.wait_limit, kSiteEpilogueTmemFull, lane);
    }
    if (have) {
        ptx::tc_fence_after();
        if (lane == 0) tr(kTrAccReady, blockIdx.x);
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16), v);
        ptx::tmem_ld_wait();
        // lane < 16 holds column n = 16 warp + lane of C, rows m0 .. m0 + NT - 1
        if (lane < 16) {
            const int n = warp * 16 + lane;
#pragma unroll
            for (int m = 0; m < NT; ++m)
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage + (uint32_t)((m * kSmallBN + n) * 4)), "r"(v[m]));
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // the accumulator is read (or never will be): its columns go back now,
        // while the stores run; every MMA completed first (the done barrier,
        // committed even after an abort)
        if (go && lane == 0 && !have) wait_drain(done_bar, 0, p.wait_limit);
        __syncwarp();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
    // an aborted launch (a wait gave up somewhere) stores nothing
    const bool store = have && *abort_flag == 0;
    if (store) {
        // NT rows of 64 columns in pieces of 16 output bytes, clipped at M and N
        // (N is a multiple of 8, so a piece is all in or all out); C += A B adds
        // C's values in fp32 first and rounds once
        constexpr int kElems = 16 / L::kOutBytes;               // outputs per piece: 8 fp16 or 4 fp32
        constexpr int kPieces = kSmallBN / kElems;              // per row
        for (int i = threadIdx.x; i < NT * kPieces; i += kSmallThreads) {
            const int m = i / kPieces, c = i % kPieces;
            const int row = m0 + m, col = n0 + c * kElems;
            if (row >= p.M || col >= p.N) continue;
            const uint32_t src = stage + (uint32_t)((m * kSmallBN + c * kElems) * 4);
            uint32_t f[8];
            ptx::ld_shared_v4(src, f[0], f[1], f[2], f[3]);
            if constexpr (OUT == 0) ptx::ld_shared_v4(src + 16, f[4], f[5], f[6], f[7]);
            const size_t off = ((size_t)row * p.N + col) * L::kOutBytes;
            if (p.c_in != nullptr) {
                const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const char*>(p.c_in) + off);
                const uint32_t h[4] = {w.x, w.y, w.z, w.w};
                if constexpr (OUT == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 g = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
                        f[2 * e] = __float_as_uint(__uint_as_float(f[2 * e]) + g.x);
                        f[2 * e + 1] = __float_as_uint(__uint_as_float(f[2 * e + 1]) + g.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) fadd_bits(f[e], h[e]);
                }
            }
            char* dst = static_cast<char*>(C) + off;
            if constexpr (OUT == 0)
                ptx::st_global_v4(dst, ptx::pack_f16x2(f[0], f[1]), ptx::pack_f16x2(f[2], f[3]),
                                  ptx::pack_f16x2(f[4], f[5]), ptx::pack_f16x2(f[6], f[7]));
            else
                ptx::st_global_v4(dst, f[0], f[1], f[2], f[3]);
        }
    }
    if (lane == 0 && store) tr(kTrStored, 0);
    if (go && threadIdx.x == 0 && p.inject == 0 && *abort_flag != 0) {
        // after an abort the producer lets every copy it issued land before the
        // CTA (and its shared memory) goes away
        for (int kb = 0; kb < KB; ++kb) wait_drain(bar0 + 8u * kb, 0, p.wait_limit);
    }
    if (lane == 0) tr(kTrExit);
}

}  // namespace tcgemm
