// Arithmetic of the kernels' on-chip allocations, shared by host and device:
// where each part of a CTA's dynamic shared memory lies, and whether an access
// stays inside the part it belongs to.  The kernels compute their shared-memory
// addresses from carve(); the bounds-check build (TCGEMM_CHECK) tests every
// ring, staging, barrier and Tensor Memory access with holds() before making
// it, and gemm_f16_check_plan (the same build, host side) runs the same tests
// over every access a plan's launch makes.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TC_HD __host__ __device__ __forceinline__
#else
#define TC_HD inline
#endif

namespace tcgemm {

// [lo, lo + size) holds all of [addr, addr + bytes)
TC_HD constexpr bool holds(uint32_t lo, uint32_t size, uint32_t addr, uint32_t bytes) {
    return addr >= lo && addr - lo <= size && bytes <= size - (addr - lo);
}

// The carve-up of a CTA's dynamic shared memory, as offsets from its first
// 1024-byte boundary (128-byte swizzle atoms sit on such boundaries): the
// ring's A parts, its B parts, 4 epilogue warps x 2 output staging buffers,
// the mbarriers, then the TMEM address slot and the abort flag (16 bytes).
struct Carve {
    uint32_t a, b, c, bar, misc, end;
};

TC_HD constexpr Carve carve(int slots, int a_bytes, int b_bytes, int staging_bytes, int num_bars) {
    Carve k{0, 0, 0, 0, 0, 0};
    k.b = (uint32_t)(slots * a_bytes);
    k.c = k.b + (uint32_t)(slots * b_bytes);
    k.bar = k.c + (uint32_t)(4 * 2 * staging_bytes);
    k.misc = k.bar + (uint32_t)(num_bars * 8);
    k.end = k.misc + 16;
    return k;
}

// Dynamic shared memory starts 16-byte aligned: rounding up to 1024 bytes
// skips at most this much.
constexpr uint32_t kMaxAlignSkip = 1024 - 16;

// Split-K blocks of the one-CTA kernel (a block: one epilogue warp's 32 rows
// of one column chunk, `block` bytes): parked in the ring at this offset from
// its start, chunk-major ...
TC_HD constexpr uint32_t park_offset(int chunk, int warp_q, uint32_t block) {
    return (uint32_t)(chunk * 4 + warp_q) * block;
}

// ... or, with two ranks, pushed into the receiving warp's two staging buffers
// at this offset from the start of all staging (each rank receives every
// second chunk).
TC_HD constexpr uint32_t push_offset(int chunk, int warp_q, uint32_t block, uint32_t staging_bytes) {
    return (uint32_t)(warp_q * 2) * staging_bytes + (uint32_t)(chunk / 2) * block;
}

}  // namespace tcgemm
