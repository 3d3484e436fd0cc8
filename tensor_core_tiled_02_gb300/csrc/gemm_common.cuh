// Pieces shared by the fp16 GEMM kernels (one CTA per tile, and the CTA pair
// of gemm_pair_kernel.cuh): tile constants, launch parameters, descriptors,
// the grouped raster, bounded mbarrier waits and the epilogue's chunk store.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "bounds.cuh"
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
    kSiteReduceData = 7,
    kSitePartialFlag = 8,
    // bounds-check build (TCGEMM_CHECK) only: an access outside its allocation
    // was about to be made, and was skipped
    kSiteSmemBounds = 9,       // shared memory: ring, staging, mbarrier, or the carve-up itself
    kSiteTmemBounds = 10,      // Tensor Memory columns beyond the CTA's allocation
    kSiteWorkspaceBounds = 11, // a stream-K workspace slot or flag beyond the plan's
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
    // stream-K: tiles [0, dp_tiles) run data-parallel; the K iterations of
    // the remaining sk_tiles are shared by the first sk_pairs clusters (CTA
    // pairs, or single CTAs in the one-CTA kernel), partial tiles meeting
    // through `ws` and `flags`.  sk_split 0: even contiguous shares.
    // sk_split > 0 (helpers, CTA pairs only): cluster c < sk_tiles runs K
    // steps [0, sk_split) of shared tile c; the H = sk_pairs - sk_tiles
    // clusters after them are helpers, helper h running steps [sk_split,
    // k_blocks) of shared tiles h, h + H, h + 2H, ... (at most sk_helper_tiles
    // of them), one unit each
    int dp_tiles, sk_tiles, sk_pairs;
    int sk_split, sk_helper_tiles;
    unsigned epoch;        // value a flag takes when its partial is ready in this launch
    float* ws;             // one 128 x 256 fp32 partial per CTA of the sharing clusters
    unsigned* flags;       // one flag per epilogue warp of those CTAs
    const void* c_in;      // accumulate into C: the values C holds before the call; NULL otherwise
    // trace build only (TCGEMM_TRACE): this launch's records, NULL when not traced;
    // trace_ctas CTAs x kTraceRoles roles x trace_events records of two words
    unsigned long long* trace;
    int trace_ctas, trace_events;
    // small launches (the pair kernel's PF instances): K steps of its first unit
    // each CTA prefetches into L2 before the dependency wait
    int pf_steps;
};

// ---- the trace build ------------------------------------------------------------
// With -DTCGEMM_TRACE, lane 0 of each role records events of its own: the
// producer (role 0), the MMA issuer (role 1) and the four epilogue warps (roles
// 2..5).  A record is two 64-bit words: the SM clock (clock64), then the event
// code (bits 63..56), its argument (bits 55..32) and, for the entry and exit
// events only, the low 32 bits of %globaltimer in nanoseconds (the one clock
// shared by all SMs, read only there: it is slow to read and ticks coarsely;
// a reader places the other events between the two by the SM clock).
// Without the define a Tracer is empty and every call vanishes.
constexpr int kTraceRoles = 6;
enum TraceEvent : unsigned {
    kTrEntry = 1,       // kernel entry (arg: SM id)
    kTrSetup = 2,       // barriers, TMEM and the cluster synchronised
    kTrDepWait = 3,     // griddepcontrol.wait returned: the previous kernel is complete
    kTrLoad = 4,        // producer issued a step's loads (arg: K step)
    kTrFull = 5,        // MMA issuer saw a step's operands land (arg: K step)
    kTrTileDone = 6,    // MMA issuer committed a unit's accumulator (arg: tile)
    kTrAccReady = 7,    // epilogue saw the accumulator complete (arg: tile)
    kTrPushed = 8,      // split-K: this warp's partials pushed to / parked for the other ranks
    kTrPartner = 9,     // split-K: the other ranks' partials of this warp's chunks are here
    kTrFlags = 10,      // stream-K owner: every contributor's flag seen
    kTrStored = 11,     // a chunk's TMA store issued (arg: chunk)
    kTrStoreRead = 12,  // the warp's stores have read their staging
    kTrExit = 13,       // the role is about to leave the kernel
    kTrParked = 14,     // stream-K contributor: partial parked and flag released
};

struct Tracer {
#ifdef TCGEMM_TRACE
    unsigned long long* rec = nullptr;
    int n = 0, cap = 0;
    __device__ __forceinline__ Tracer(const KernelParams& p, int role) {
        if (p.trace != nullptr && (int)blockIdx.x < p.trace_ctas) {
            rec = p.trace + 2ull * ((unsigned long long)(blockIdx.x * kTraceRoles + role) * p.trace_events);
            cap = p.trace_events;
        }
    }
    __device__ __forceinline__ void operator()(unsigned code, unsigned arg = 0) {
        if (rec == nullptr || n >= cap) return;
        const unsigned long long clk = clock64();
        const unsigned gt = (code == kTrEntry || code == kTrExit) ? (unsigned)ptx::globaltimer() : 0u;
        rec[2 * n] = clk;
        rec[2 * n + 1] = ((unsigned long long)code << 56) | ((unsigned long long)(arg & 0xFFFFFFu) << 32) | gt;
        ++n;
    }
#else
    __device__ __forceinline__ Tracer(const KernelParams&, int) {}
    __device__ __forceinline__ void operator()(unsigned, unsigned = 0) {}
#endif
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
    // full[8], empty[8], tmem_full[2], tmem_empty[2], drain, red_ready, red_data, dry
    static constexpr int kNumBars = 2 * kMaxStages + 8;
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
// Every second group walks the n-blocks backwards (a serpentine), so a group
// starts on the columns of B the group before it ended on, still in L2.
__device__ __forceinline__ void tile_coords(int t, const KernelParams& p, int& mb, int& nb) {
    const int g = p.raster_group;
    const int per_group = g * p.tiles_n;
    const int grp = t / per_group;
    const int first_m = grp * g;
    const int gm = min(p.tiles_m - first_m, g);
    const int r = t - grp * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
    if (grp & 1) nb = p.tiles_n - 1 - nb;
}

__device__ __forceinline__ void record_timeout(unsigned site) { atomicCAS(&g_status, 0u, site); }

// The bounds-check build tests an access before making it; a failed test
// records its site (first writer wins), raises the CTA's abort flag (every
// bounded wait then gives up) and the caller skips the access.  Without
// TCGEMM_CHECK the test is the constant true and vanishes.
#ifdef TCGEMM_CHECK
__device__ __forceinline__ bool bounds_ok(bool ok, unsigned site, volatile int* abort_flag) {
    if (ok) return true;
    record_timeout(site);
    *abort_flag = 1;
    return false;
}
#define TC_CHECK(cond, site) bounds_ok((cond), (site), abort_flag)
#else
#define TC_CHECK(cond, site) true
#endif

constexpr int kPartialFloats = kBM * 256;  // one CTA's fp32 partial tile (up to 128 x 256) in the workspace
constexpr int kMaxSkCtas = 1024;           // CTAs whose flags the workspace's fixed flag area holds (4 each)

// The units of work of one cluster (a CTA pair, or a single CTA): its share
// of the stream-K iterations first, then its data-parallel tiles c,
// c + clusters, ... below dp_tiles.  Running the shares first keeps every
// sharing cluster on the same K range at the same time, and an owner unit's
// wait for its contributors' partials, and their reduction, overlap the
// cluster's next tile instead of ending the launch.  Under helper stream-K
// the main units (steps [0, sk_split) of one shared tile each) run in step
// with one another, and so do the helpers (steps [sk_split, k_blocks) of one
// tile after another, the helpers' j-th tiles being H consecutive ones): at
// any time two K ranges are in use, whose operand blocks the sharing pairs
// find in L2.  Producer, MMA issuer and epilogue walk the same sequence.
struct UnitIter {
    int next_dp, stride;
    long long it, it_end;  // even shares: flat (tile, K step) iterations; main, helper: local tile indices
    int ndp;      // data-parallel units handed out so far
    int sk_kind;  // 0 even share, 1 main unit, 2 helper units (local tiles it, it + H, ...)
};

// First stream-K iteration of cluster c: the sk_tiles * k_blocks iterations
// are dealt out in sk_pairs contiguous, equal (to one) shares.
__device__ __forceinline__ long long sk_begin(const KernelParams& p, int c) {
    return (long long)p.sk_tiles * p.k_blocks * c / p.sk_pairs;
}

__device__ __forceinline__ void unit_iter_init(UnitIter& u, const KernelParams& p, int c, int clusters) {
    u.next_dp = c;
    u.stride = clusters;
    u.ndp = 0;
    u.sk_kind = 0;
    u.it = u.it_end = 0;
    if (p.sk_tiles > 0 && c < p.sk_pairs) {
        if (p.sk_split == 0) {
            u.it = sk_begin(p, c);
            u.it_end = sk_begin(p, c + 1);
        } else if (c < p.sk_tiles) {
            u.sk_kind = 1;
            u.it = c;
            u.it_end = c + 1;
        } else {
            u.sk_kind = 2;
            u.it = c - p.sk_tiles;
            u.it_end = p.sk_tiles;
        }
    }
}

__device__ __forceinline__ void sk_unit(UnitIter& u, const KernelParams& p, int& tile, int& k0, int& k1) {
    const int KB = p.k_blocks;
    if (u.sk_kind != 0) {
        tile = p.dp_tiles + (int)u.it;
        k0 = u.sk_kind == 1 ? 0 : p.sk_split;
        k1 = u.sk_kind == 1 ? p.sk_split : KB;
        u.it += u.sk_kind == 1 ? 1 : p.sk_pairs - p.sk_tiles;
        return;
    }
    const int local = (int)(u.it / KB);
    k0 = (int)(u.it - (long long)local * KB);
    const long long left = u.it_end - u.it;
    k1 = left < (long long)(KB - k0) ? k0 + (int)left : KB;
    tile = p.dp_tiles + local;
    u.it += k1 - k0;
}

// Workspace slot of the partial a contributor unit of tile t parks (cluster
// c's, which runs that unit): its cluster under even shares, the tile under
// helpers (a helper contributes to several tiles, each tile has one helper).
__device__ __forceinline__ int sk_park_slot(const KernelParams& p, int c, int t) {
    return p.sk_split > 0 ? t - p.dp_tiles : c;
}

// Slots [first, end) whose partials the owner unit of tile t (cluster c's)
// adds to its own, in this order: under even shares the following clusters
// whose shares start inside the tile, under helpers the tile's one slot.
__device__ __forceinline__ void sk_owner_slots(const KernelParams& p, int c, int t, int& first, int& end) {
    if (p.sk_split > 0) {
        first = t - p.dp_tiles;
        end = first + 1;
        return;
    }
    first = end = c + 1;
    const long long tile_end = (long long)(t - p.dp_tiles + 1) * p.k_blocks;
    while (end < p.sk_pairs && sk_begin(p, end) < tile_end) ++end;
}

// Workspace slots of this plan (partials of CTA pairs take two each).
__device__ __forceinline__ int sk_slots(const KernelParams& p) { return p.sk_split > 0 ? p.sk_tiles : p.sk_pairs; }

// Next unit: tile id and K-step range [k0, k1).  False when none is left.
__device__ __forceinline__ bool unit_next(UnitIter& u, const KernelParams& p, int& tile, int& k0, int& k1) {
    if (u.it < u.it_end) {
        sk_unit(u, p, tile, k0, k1);
        return true;
    }
    if (u.next_dp < p.dp_tiles) {
        tile = u.next_dp;
        u.next_dp += u.stride;
        ++u.ndp;
        k0 = 0;
        k1 = p.k_blocks;
        return true;
    }
    return false;
}

// Bounded wait until a flag holds this launch's epoch (acquire).
__device__ __forceinline__ bool wait_flag(const unsigned* f, unsigned epoch, volatile int* abort_flag,
                                          long long limit) {
    if (ptx::ld_acquire_gpu(f) == epoch) return true;
    const long long t0 = clock64();
    while (ptx::ld_acquire_gpu(f) != epoch) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            record_timeout(kSitePartialFlag);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

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

// One 128-byte-wide column chunk of a warp's 32 output rows into staging
// buffer `stg` (4 KiB, 1024-byte aligned) that no earlier store of this warp
// still reads: convert, write it in the 128-byte swizzle the C tensor map
// expects (16-byte chunk j of row `lane` at chunk j ^ (lane % 8)), fence for
// the async proxy and TMA-store it.  skip_store: everything but the TMA store
// itself.  Returns whether a store was issued.  The last tile of a CTA drains
// through its idle operand ring, one buffer per chunk and nothing waited for
// (store_chunk with a ring buffer).
template <int OUT>
__device__ __forceinline__ bool stage_and_store(const uint32_t (&v)[OUT == 0 ? 64 : 32], const CUtensorMap* tmC,
                                                uint32_t stg, int lane, int x, int y, bool skip_store = false) {
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
    if (skip_store) return false;
    if (lane == 0) {
        ptx::tma_store_2d(tmC, stg, x, y);
        ptx::bulk_commit_group();
    }
    return true;
}

// stage_and_store through the warp's two staging buffers in turn (nstore
// counts its stores), waiting first for the store issued from the buffer two
// rounds ago to have read it; or, with ring_buf != 0, through that buffer of
// the idle operand ring, waiting for nothing (the same instructions either
// way, so a dry pass through one warms the other).  skip_store: everything but
// the TMA store itself (and nstore stays).  A dry pass through the drain
// normally stores instead to rows from M on, which the tensor map clips
// entirely: no byte of C is written.
template <int OUT>
__device__ __forceinline__ void store_chunk(const uint32_t (&v)[OUT == 0 ? 64 : 32], const CUtensorMap* tmC,
                                            uint32_t staging, int& nstore, int lane, int x, int y,
                                            bool skip_store = false, uint32_t ring_buf = 0) {
    const uint32_t stg = ring_buf != 0 ? ring_buf : staging + (uint32_t)((nstore & 1) * 4096);
    // the store issued from this buffer two rounds ago must have read it
    if (ring_buf == 0 && lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
    if (stage_and_store<OUT>(v, tmC, stg, lane, x, y, skip_store)) ++nstore;
}

__device__ __forceinline__ void fadd_bits(uint32_t& acc, uint32_t add) {
    acc = __float_as_uint(__uint_as_float(acc) + __uint_as_float(add));
}

// Accumulating into C: add to a lane's chunk (row `row`, columns x .. x+127
// bytes) the values C holds there before this call, in fp32.  The lane that
// stores the chunk reads it first, so no other thread touches those elements.
// Rows past M and 16-byte column groups past N (N % 8 == 0) are skipped.
template <int OUT>
__device__ __forceinline__ void add_c_in(uint32_t (&v)[OUT == 0 ? 64 : 32], const KernelParams& p, int row, int x) {
    if (p.c_in == nullptr || row >= p.M) return;
    constexpr int kPer16 = OUT == 0 ? 8 : 4;  // elements in 16 bytes
    const char* base = static_cast<const char*>(p.c_in) + ((size_t)row * p.N + x) * (OUT == 0 ? 2 : 4);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (x + j * kPer16 >= p.N) break;
        const uint4 w = *reinterpret_cast<const uint4*>(base + j * 16);
        if constexpr (OUT == 0) {
            const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
                v[8 * j + 2 * e] = __float_as_uint(__uint_as_float(v[8 * j + 2 * e]) + f.x);
                v[8 * j + 2 * e + 1] = __float_as_uint(__uint_as_float(v[8 * j + 2 * e + 1]) + f.y);
            }
        } else {
            fadd_bits(v[4 * j], w.x);
            fadd_bits(v[4 * j + 1], w.y);
            fadd_bits(v[4 * j + 2], w.z);
            fadd_bits(v[4 * j + 3], w.w);
        }
    }
}

}  // namespace tcgemm
