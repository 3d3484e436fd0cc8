// The pipelined blocked add Z = X + Y (f32) on the GEMM's pipeline machinery.
//
// Method ("JAX Pallas 软件流水线 Software Pipelining 完全指南", sections 4 and
// 6): the arrays are cut into blocks; each step copies one block of X and one
// of Y from HBM into fast memory, adds them, and copies the block of Z back,
// with the copies of the next blocks in flight while the current one is
// added.  Here the blocks are 32 x 256 tiles walked by persistent CTAs:
//   warp 0       one lane TMA-loads X and Y tiles into a ring of `slots`
//                shared-memory buffers (mbarrier `full`, expect-tx)
//   warps 1..4   each adds its 8 rows of the tile in place (one IEEE binary32
//                addition per element, round to nearest even), TMA-stores
//                them to Z and, once that store has read the buffer, arrives
//                on the slot's `empty` barrier (4 arrivals free the slot)
// The blocking changes no element's arithmetic: Z is bit-exact X + Y.  Ragged
// edges: TMA zero-fills loads past M or N and clips the stores.
// Waits are bounded as in the GEMM kernels (status word, abort flag).
#pragma once

#include "gemm_common.cuh"

namespace tcgemm {

constexpr int kAddBM = 32;                          // tile rows
constexpr int kAddBN = 256;                         // tile columns (f32): the longest TMA box side
constexpr int kAddWarps = 4;                        // consumer warps, kAddBM / 4 rows each
constexpr int kAddThreads = 32 * (1 + kAddWarps);
constexpr int kAddTileBytes = kAddBM * kAddBN * 4;  // 32 KiB per operand tile
constexpr int kAddMaxSlots = 4;

struct AddParams {
    int M, N;
    int tiles_m, tiles_n;
    int slots;
    long long wait_limit;
};

struct AddLayout {
    static constexpr int kNumBars = 2 * kAddMaxSlots;
    static constexpr int smem_bytes(int slots) { return slots * 2 * kAddTileBytes + kNumBars * 8 + 16 + 1024; }
};

__global__ void __launch_bounds__(kAddThreads, 1)
    add_f32_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                   const __grid_constant__ CUtensorMap tmZ, const AddParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int S = p.slots;
    const uint32_t sX = base;
    const uint32_t sY = sX + S * kAddTileBytes;
    const uint32_t bar0 = sY + S * kAddTileBytes;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + (bar0 - base) + AddLayout::kNumBars * 8);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kAddMaxSlots + s); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), kAddWarps);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmY);
        ptx::prefetch_tmap(&tmZ);
    }
    __syncthreads();
    // each role waits for the previous kernel in the stream just before its
    // first global-memory access: the producer before its first load (its
    // set-up runs earlier, overlapping that kernel), the adding warps before
    // their first store

    const int num_tiles = p.tiles_m * p.tiles_n;
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool dep_done = false;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit, kSiteProducerEmpty)) break;
                const int x = (t % p.tiles_n) * kAddBN;
                const int y = (t / p.tiles_n) * kAddBM;
                const uint32_t fb = full_bar(stage);
                ptx::mbar_arrive_expect_tx(fb, 2 * kAddTileBytes);
                if (!dep_done) {
                    ptx::grid_dependency_wait();
                    ptx::grid_launch_dependents();
                    dep_done = true;
                }
                ptx::tma_load_2d(sX + stage * kAddTileBytes, &tmX, fb, x, y);
                ptx::tma_load_2d(sY + stage * kAddTileBytes, &tmY, fb, x, y);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // every load lands before shared memory goes away
            for (int s = 0; s < S; ++s)
                if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_phase >> s) & 1u, p.wait_limit);
        }
    } else {
        ptx::grid_dependency_wait();
        ptx::grid_launch_dependents();
        const int w = warp - 1;               // this warp's rows: 8w .. 8w+7 of the tile
        constexpr int kRows = kAddBM / kAddWarps;
        constexpr int kVec = kRows * kAddBN / 4 / 32;  // 16-byte groups per lane
        int stage = 0, prev = -1;
        uint32_t phase = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            if (!warp_wait(full_bar(stage), phase, abort_flag, 4 * p.wait_limit, kSiteMmaFull, lane)) break;
            const uint32_t xs = sX + stage * kAddTileBytes + w * kRows * kAddBN * 4;
            const uint32_t ys = sY + stage * kAddTileBytes + w * kRows * kAddBN * 4;
#pragma unroll
            for (int i = 0; i < kVec; ++i) {
                // consecutive lanes, consecutive 16 bytes: no bank conflicts
                const uint32_t off = (uint32_t)((i * 32 + lane) * 16);
                float a0, a1, a2, a3, b0, b1, b2, b3;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                             : "r"(xs + off));
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3)
                             : "r"(ys + off));
                ptx::st_shared_v4(xs + off, __float_as_uint(__fadd_rn(a0, b0)), __float_as_uint(__fadd_rn(a1, b1)),
                                  __float_as_uint(__fadd_rn(a2, b2)), __float_as_uint(__fadd_rn(a3, b3)));
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d(&tmZ, xs, (t % p.tiles_n) * kAddBN, (t / p.tiles_n) * kAddBM + w * kRows);
                ptx::bulk_commit_group();
                // the previous tile's store has read its buffer: free that slot
                ptx::bulk_wait_group_read<1>();
                if (prev >= 0) ptx::mbar_arrive(empty_bar(prev));
            }
            __syncwarp();
            prev = stage;
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0) {
            ptx::bulk_wait_group_read<0>();
            if (prev >= 0) ptx::mbar_arrive(empty_bar(prev));
        }
        __syncwarp();
    }
    __syncthreads();
}

}  // namespace tcgemm
