// Host side of the fp16 GEMM: argument checks, the planner, tensor-map
// encoding and the launch.  The C ABI is declared in include/gemm_f16.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "add_matrices.h"
#include "gemm_f16.h"
#ifdef TCGEMM_TRACE
#include "gemm_f16_trace.h"
#endif
#ifdef TCGEMM_CHECK
#include "gemm_f16_check.h"
#endif
#include "add_kernel.cuh"
#include "gemm_kernel.cuh"
#include "gemm_pair_kernel.cuh"
#include "gemm_small_kernel.cuh"

namespace {

using namespace tcgemm;

constexpr int kMaxDevices = 64;
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_100-class parts
constexpr long long kDefaultWaitLimit = 2000000000LL;  // ~1 s at 2 GHz
constexpr int kMinHelperSteps = 8;  // helper stream-K: fewest K steps of a tile a helper pair runs
constexpr int kMaxHelperTiles = 8;  // helper stream-K: most tiles one helper pair runs
constexpr int kPrefetchSteps = 8;   // small pair launches: K steps each CTA prefetches into L2

std::mutex g_mu;
gemm_config g_cfg = {};

// Per-device facts, filled on first use.  Fast paths read the atomics; the
// first fill of each takes g_dev_mu, so concurrent first calls from several
// host threads are safe.
struct DeviceInfo {
    std::atomic<bool> ready{false};
    int sms = 0;
    int cc = 0;
    std::atomic<int> max_pairs{0};  // CTA-pair clusters the GPU holds at once (0: not yet asked)
    // [s]: clusters of s one-CTA-per-SM CTAs of the one-CTA kernel the GPU holds at once (0: not yet asked)
    std::atomic<int> max_clusters[kMaxSplit + 1];
    // [tile_n 64 / 128 / 256, 256 x 256 CTA pair with step K 64 / 128, blocked add,
    // 128 x 128 CTA pair, its prefetching instance, small kernel of 8 / 16 / 32
    // rows][out_dtype]: the kernel's shared-memory limit has been raised on this
    // device
    std::atomic<bool> attr_set[11][2];
};
DeviceInfo g_dev[kMaxDevices];  // static storage: every atomic starts zero
std::mutex g_dev_mu;

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename Kern>
int ensure_smem_limit(Kern kern, int bytes, std::atomic<bool>& done) {
    if (done.load(std::memory_order_acquire)) return GEMM_OK;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!done.load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        done.store(true, std::memory_order_release);
    }
    return GEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<unsigned> g_epoch{0};  // stream-K flag value of the latest launch
std::once_flag g_encode_once;

int out_bytes(int out_dtype) { return out_dtype == GEMM_OUT_F16 ? 2 : 4; }

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Argument checks that need no CUDA.  Returns GEMM_OK, or 1 for "nothing to do".
int check_args(const void* A, const void* B, const void* C, int M, int N, int K, int out_dtype, bool check_ptrs) {
    if (out_dtype != GEMM_OUT_F16 && out_dtype != GEMM_OUT_F32) return GEMM_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_DIM;
    if (N % 8 != 0 || K % 8 != 0) return GEMM_ERR_ALIGN;
    // tile ids and tile coordinates must fit an int, for the narrowest tile (64 columns)
    if ((long long)ceil_div(M, kBM) * ceil_div(N, 64) > INT_MAX) return GEMM_ERR_DIM;
    if (M == 0 || N == 0) return 1;
    if (!check_ptrs) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_NULL;
    const uintptr_t a = (uintptr_t)A, b = (uintptr_t)B, c = (uintptr_t)C;
    if ((c & 15) || (K > 0 && ((a & 15) || (b & 15)))) return GEMM_ERR_ALIGN;
    if (K > 0) {
        // inputs read-only, output write-only: C may not overlap A or B
        const uint64_t c_end = c + (uint64_t)M * N * out_bytes(out_dtype);
        const uint64_t a_end = a + (uint64_t)M * K * 2;
        const uint64_t b_end = b + (uint64_t)K * N * 2;
        if (c < a_end && a < c_end) return GEMM_ERR_ALIAS;
        if (c < b_end && b < c_end) return GEMM_ERR_ALIAS;
    }
    return GEMM_OK;
}

int check_config(const gemm_config& c) {
    if (c.tile_n != 0 && c.tile_n != 64 && c.tile_n != 128 && c.tile_n != 256) return GEMM_ERR_CONFIG;
    if (c.stages < 0 || c.stages > kMaxStages) return GEMM_ERR_CONFIG;
    if (c.release < 0 || c.release >= kMaxStages) return GEMM_ERR_CONFIG;
    if (c.stages != 0 && c.release >= c.stages) return GEMM_ERR_CONFIG;
    if (c.stages + c.release > kMaxStages) return GEMM_ERR_CONFIG;
    if (c.grid < 0 || c.raster_group < 0 || c.wait_limit < 0) return GEMM_ERR_CONFIG;
    if (c.inject_stall != 0 && c.inject_stall != 1) return GEMM_ERR_CONFIG;
    if (c.split < 0 || c.split > kMaxSplit) return GEMM_ERR_CONFIG;
    if (c.cta_group < 0 || c.cta_group > 2) return GEMM_ERR_CONFIG;
    // CTA pairs: tile_n 0 or 256 for 256 x 256 tiles, 128 for 128 x 128 tiles
    if (c.cta_group == 2 && ((c.tile_n != 0 && c.tile_n != 128 && c.tile_n != 256) || c.split > 1))
        return GEMM_ERR_CONFIG;
    if (c.tile_k != 0 && c.tile_k != 64 && c.tile_k != 128) return GEMM_ERR_CONFIG;
    if (c.stream_k < 0 || c.stream_k > 2) return GEMM_ERR_CONFIG;
    return GEMM_OK;
}

int smem_for(int tile_n, int out_dtype, int slots) {
    if (tile_n == 256)
        return out_dtype == GEMM_OUT_F16 ? Layout<256, 0>::smem_bytes(slots) : Layout<256, 1>::smem_bytes(slots);
    if (tile_n == 64)
        return out_dtype == GEMM_OUT_F16 ? Layout<64, 0>::smem_bytes(slots) : Layout<64, 1>::smem_bytes(slots);
    return out_dtype == GEMM_OUT_F16 ? Layout<128, 0>::smem_bytes(slots) : Layout<128, 1>::smem_bytes(slots);
}

// Shared memory to request so that no SM ever holds more CTAs of this launch
// than its 512 TMEM columns serve at once: a CTA of a cluster left waiting in
// tcgen05.alloc for columns held by another cluster's CTA could otherwise
// wait on a peer that waits in turn.  (228 KiB of shared memory per SM.)
int smem_request(int smem_bytes, int tmem_cols) {
    const int max_ctas = 512 / tmem_cols;
    const int floor_bytes = 233472 / (max_ctas + 1) + 1;
    return smem_bytes > floor_bytes ? smem_bytes : floor_bytes;
}

// pair_m: the pair's tile, 256 (256 x 256) or 128 (128 x 128, 128-deep steps only)
int smem_for_pair(int out_dtype, int step_k, int pair_m, int slots) {
    if (pair_m == 128)
        return out_dtype == GEMM_OUT_F16 ? PairLayout<0, 128, 128, 128>::smem_bytes(slots)
                                         : PairLayout<1, 128, 128, 128>::smem_bytes(slots);
    if (step_k == 128)
        return out_dtype == GEMM_OUT_F16 ? PairLayout<0, 128>::smem_bytes(slots)
                                         : PairLayout<1, 128>::smem_bytes(slots);
    return out_dtype == GEMM_OUT_F16 ? PairLayout<0, 64>::smem_bytes(slots) : PairLayout<1, 64>::smem_bytes(slots);
}

int smem_for_small(int out_dtype, int rows, int k_blocks) {
    if (out_dtype == GEMM_OUT_F16)
        return rows == 8 ? SmallLayout<0, 8>::smem_bytes(k_blocks)
               : rows == 16 ? SmallLayout<0, 16>::smem_bytes(k_blocks) : SmallLayout<0, 32>::smem_bytes(k_blocks);
    return rows == 8 ? SmallLayout<1, 8>::smem_bytes(k_blocks)
           : rows == 16 ? SmallLayout<1, 16>::smem_bytes(k_blocks) : SmallLayout<1, 32>::smem_bytes(k_blocks);
}

// Small problems, under the default config only: the rows of C per CTA of
// the small kernel (one CTA per rows x 64 tile, every K step loaded at once,
// so K <= 1024): the fewest of 8, 16, 32 that keep the tiles within one
// wave; 0 when the small kernel does not take the problem.
int small_rows(int M, int N, int K, int num_sms, const gemm_config& cfg) {
    if (cfg.tile_n || cfg.cta_group || cfg.split || cfg.stream_k || cfg.grid || cfg.tile_k || cfg.stages ||
        cfg.release)
        return 0;
    if (M <= 0 || N <= 0 || K <= 0 || ceil_div(K, 64) > kSmallMaxKB) return 0;
    const long long cols = ceil_div(N, kSmallBN);
    for (int rows : {8, 16, 32})
        if ((long long)ceil_div(M, rows) * cols <= num_sms) return rows;
    return 0;
}

int max_slots_for(int tile_n, int out_dtype) {
    int s = kMaxStages;
    while (s > 1 && smem_for(tile_n, out_dtype, s) > kSmemLimit) --s;
    return s;
}

int max_slots_for_pair(int out_dtype, int step_k, int pair_m) {
    int s = kMaxStages;
    while (s > 1 && smem_for_pair(out_dtype, step_k, pair_m, s) > kSmemLimit) --s;
    return s;
}

// Workspace of a stream-K plan shared by `ctas` CTAs: a flag per epilogue
// warp of up to kMaxSkCtas CTAs, then one fp32 partial of up to 128 x 256 per
// CTA.  The flag area has the same size in every plan, so a flag word never
// lies where another plan keeps a partial tile: it only ever holds 0 or the
// epoch of some launch.
constexpr size_t kFlagBytes = (size_t)kMaxSkCtas * 4 * sizeof(unsigned);  // 16 KiB

constexpr size_t workspace_for(int ctas) { return kFlagBytes + (size_t)ctas * kPartialFloats * sizeof(float); }

// Clusters the GPU can hold at once, by cluster size (one CTA per SM): [1] the
// SMs, [2] CTA pairs, [3 .. kMaxSplit] split-K clusters.  Not every size packs
// the SMs: on a 152-SM GB300 they are 76, 46, 36, 28, 23, 15 and 15 clusters
// of 2 .. 8 (a cluster's CTAs share a GPC).  A split-K launch whose clusters do
// not all fit at once runs in two waves.
struct Fit {
    int clusters[kMaxSplit + 1];
};

// For planning without the device at hand: the 152-SM GB300 figures, scaled
// to `num_sms`.
Fit fit_estimate(int num_sms) {
    static const int kGb300[kMaxSplit + 1] = {0, 152, 76, 46, 36, 28, 23, 15, 15};
    Fit f;
    f.clusters[0] = 0;
    for (int c = 1; c <= kMaxSplit; ++c) f.clusters[c] = (int)((long long)kGb300[c] * num_sms / 152);
    if (f.clusters[2] < 1 && num_sms >= 2) f.clusters[2] = 1;
    return f;
}

// The planner.
// CTA pairs with 256 x 256 tiles for large problems (see the cta_group choice
// below); CTA pairs with 128 x 128 tiles for small ones whose tiles fit one
// wave of pairs without splitting K.  Otherwise one CTA per tile:
// Tile: 128 x 256 or 128 x 128, whichever needs less time counted in waves of
// tiles over the SMs, a 128 x 128 tile costing 0.85 of a 128 x 256 one (half
// the MMA work at about 0.6 of the tensor-pipe efficiency, measured: it needs
// the whole shared-memory port per SM).  128 x 64 is only taken on request.
// Split-K: when the tiles fill less than half the SMs, a cluster of `split`
// CTAs shares each tile along K (at least 16 K steps each), one tile per cluster.
// Pipeline depth, in the pages' terms: `stages` (max_concurrent_steps) loads in
// flight ahead of the MMA and `release` (delay_release) extra steps before a
// buffer is handed back, so the ring holds stages + release buffers.  As in
// emit_pipeline, stages must exceed release, and stages is clamped to the
// steps one CTA runs (never below release + 1).  Default: the deepest ring
// that fits shared memory.
int plan_impl(int M, int N, int K, int out_dtype, int num_sms, const Fit& fit, bool with_workspace,
              const gemm_config& cfg, gemm_plan* p) {
    std::memset(p, 0, sizeof(*p));
    if (const int rows = small_rows(M, N, K, num_sms, cfg)) {
        p->cta_group = 1;
        p->tile_m = rows;
        p->tile_n = kSmallBN;
        p->tile_k = 64;
        p->tiles_m = ceil_div(M, rows);
        p->tiles_n = ceil_div(N, kSmallBN);
        p->num_tiles = p->tiles_m * p->tiles_n;
        p->k_steps = ceil_div(K, 64);
        p->stages = p->slots = p->k_steps;  // every K block in flight at once
        p->split = 1;
        p->grid = p->num_tiles;
        p->raster_group = 1;
        p->dp_tiles = p->num_tiles;
        p->tmem_cols = 32;
        p->smem_bytes = smem_request(smem_for_small(out_dtype, rows, p->k_steps), p->tmem_cols);
        p->threads = kSmallThreads;
        return GEMM_OK;
    }
    int max_pairs = fit.clusters[2];
    p->tile_m = kBM;
    p->tile_k = kBK;
    const int tiles_m = ceil_div(M, kBM);
    int tn = cfg.tile_n;
    bool wide_to_split = false;
    if (tn == 0) {
        const long long t256 = (long long)tiles_m * ceil_div(N, 256);
        const long long t128 = (long long)tiles_m * ceil_div(N, 128);
        const long long w256 = (t256 + num_sms - 1) / num_sms;
        const long long w128 = (t128 + num_sms - 1) / num_sms;
        tn = w256 * 100 <= w128 * 85 ? 256 : 128;
        // Each SM takes in at most about 100 GB/s of operands from L2, so a
        // one-CTA tile's time goes with the bytes it loads: per K step 32 KiB
        // for a 128 x 128 tile, 48 KiB for twice the work on 128 x 256.  When
        // 128 x 128 tiles would fill more than half the SMs, and so run
        // unsplit, but 128 x 256 tiles leave room to split K two ways, the wide
        // split tiles load 3/4 of the bytes per CTA on as many CTAs:
        // 512 x 4096 x 8192 measured 45.1 -> 31.6 us, 256 x 8192 x 8192 45.4
        // -> 35.0 us (CTA pairs with a stream-K tail: 35.4 and 40.3 us).
        if (tn == 128 && cfg.split == 0 && cfg.stream_k != 2 && 2 * t128 > num_sms && 2 * t256 <= num_sms &&
            ceil_div(K, kBK) / 16 >= 2) {
            tn = 256;
            wide_to_split = true;
        }
    }
    p->tile_n = tn;
    p->tiles_m = tiles_m;
    p->tiles_n = ceil_div(N, tn);
    p->num_tiles = p->tiles_m * p->tiles_n;
    p->k_steps = ceil_div(K, kBK);

    // CTA pair (cta_group::2, 256 x 256 tiles on two SMs): when the wide tile
    // wins and no split is wanted, if its waves cost no more than 1/0.9 of the
    // single-CTA waves (it moves a third less operand data per SM and step).
    int cg = cfg.cta_group;
    int pm = cg == 2 && cfg.tile_n == 128 ? 128 : 256;  // CTA pairs: 256 x 256 or 128 x 128 tiles
    if (cg == 0) {
        cg = 1;
        const long long tiles128 = (long long)tiles_m * ceil_div(N, 128);
        if (tn == 256 && !wide_to_split && cfg.tile_n == 0 && cfg.split <= 1 && p->k_steps > 0 && num_sms >= 2) {
            const long long pair_tiles = (long long)ceil_div(M, 2 * kBM) * ceil_div(N, 256);
            const long long w_pair = (pair_tiles + num_sms / 2 - 1) / (num_sms / 2);
            const long long w_one = ((long long)p->num_tiles + num_sms - 1) / num_sms;
            if (w_pair * 9 <= w_one * 10 && 2 * tiles128 > num_sms) cg = 2;
        }
        // Small problems: 128 x 128 tiles on CTA pairs (M = 128 over two SMs,
        // 64 rows each) when they all fit one wave of pairs and one-CTA tiles
        // would not split K: twice the CTAs of one-CTA tiles, each loading half
        // the operands.  Not where split-K applies: streaming B from HBM (one
        // row of tiles, N = K = 8192) the pair tiles took 33.7 us against
        // 27.5 us for split-K over two CTAs (each pair steps in lock-step on
        // both SMs' loads, and each CTA reads B rows 128 bytes at a time).
        if (cg == 1 && cfg.tile_n == 0 && cfg.split == 0 && cfg.grid == 0 && cfg.stream_k != 2 &&
            p->k_steps > 0 && num_sms >= 2 && tiles128 <= max_pairs) {
            long long split1 = 1;
            if (2 * tiles128 <= num_sms) {
                split1 = num_sms / tiles128;
                if (split1 > kMaxSplit) split1 = kMaxSplit;
                if (split1 > p->k_steps / 16) split1 = p->k_steps / 16;
            }
            if (split1 <= 1) {
                cg = 2;
                pm = 128;
            }
        }
    }
    if (cg == 2) {
        if (p->k_steps == 0 || num_sms < 2) return GEMM_ERR_CONFIG;
        // 128-deep steps (eight MMAs per barrier wait and commit) unless K is
        // short; 128 x 128 pair tiles always take 128-deep steps
        if (pm == 128 && cfg.tile_k != 0 && cfg.tile_k != 128) return GEMM_ERR_CONFIG;
        const int sk = pm == 128 ? 128 : cfg.tile_k > 0 ? cfg.tile_k : (K >= 256 ? 128 : kBK);
        p->cta_group = 2;
        p->tile_k = sk;
        p->k_steps = ceil_div(K, sk);
        p->tile_m = pm;
        p->tile_n = pm;
        p->tiles_m = ceil_div(M, pm);
        p->tiles_n = ceil_div(N, pm);
        p->num_tiles = p->tiles_m * p->tiles_n;
        p->split = 1;
        if (cfg.grid > 0 && cfg.grid / 2 < max_pairs) max_pairs = cfg.grid / 2 > 0 ? cfg.grid / 2 : 1;
        int pairs = p->num_tiles < max_pairs ? p->num_tiles : max_pairs;
        // Stream-K (needs a workspace): when the last wave of tiles would leave
        // pairs idle, each of its R tiles is split along K into s equal parts,
        // s = pairs / R (2..4, at least 8 K steps a part), run by s * R pairs at
        // once.  Equal parts keep the pairs that hold part j of different tiles
        // on the same K range at the same time, so tiles sharing a row block of
        // A or a column block of B still share it in L2.  When the last wave is
        // more than half full (no two parts fit), the R tiles run their first
        // sk_split steps on R pairs in step with one another while the pairs
        // idle in that wave, as helpers, run the remaining steps of up to m
        // tiles each, one tile after another and in step with one another too.
        // Each tile then meets one helper's partial.  Helpers run a little
        // slower per step (operands less shared in L2, a pipeline refill per
        // tile, the partial to park), so they get 10 % less than an even split:
        // steps - sk_split = 0.9 steps / (m + 1).  Shared units run first; the
        // full waves, data-parallel, follow (1024 x 8192 x 8192: 85.7 -> 82.7
        // us).  Even shares of the last wave over all pairs instead start the
        // pairs at scattered K offsets, lose the L2 sharing and gain nothing.
        // stream_k 2 (testing) shares every tile's iterations evenly over all
        // pairs instead.
        p->dp_tiles = p->num_tiles;
        int sk_tiles = 0, sk_pairs = 0, clusters = pairs, sk_split = 0, sk_helper = 0;
        if (cfg.stream_k == 2) {
            clusters = max_pairs < kMaxSkCtas / 2 ? max_pairs : kMaxSkCtas / 2;
            sk_tiles = p->num_tiles;
            const long long iters = (long long)sk_tiles * p->k_steps;
            sk_pairs = (int)(iters < clusters ? iters : clusters);
        } else if (cfg.stream_k == 0) {
            const int R = p->num_tiles < max_pairs ? p->num_tiles : p->num_tiles % pairs;
            if (R > 0) {
                int parts = max_pairs / R;
                if (parts > 4) parts = 4;
                if (parts > p->k_steps / 8) parts = p->k_steps / 8;
                if (parts >= 2 && 2 * parts * R <= kMaxSkCtas) {
                    sk_tiles = R;
                    sk_pairs = parts * R;
                    clusters = p->num_tiles < max_pairs ? sk_pairs : pairs;
                } else if (parts < 2 && 2 * R <= kMaxSkCtas) {
                    const int KB = p->k_steps;
                    const int m = ceil_div(R, max_pairs - R);
                    const int l = (int)(0.9 * KB / (m + 1));
                    // worth it only with at least kMinHelperSteps steps a helper unit,
                    // few units a helper, and the wave at least 5 % shorter
                    if (l >= kMinHelperSteps && m <= kMaxHelperTiles && (long long)(KB - l) * 100 <= (long long)KB * 95) {
                        sk_tiles = R;
                        sk_split = KB - l;
                        sk_helper = m;
                        sk_pairs = R + ceil_div(R, m);
                        clusters = p->num_tiles < max_pairs ? sk_pairs : pairs;
                    }
                }
            }
        }
        if (sk_tiles > 0) {
            // partial slots: one per sharing pair, or one per tile under helpers
            p->workspace_bytes = (long long)workspace_for(2 * (sk_split > 0 ? sk_tiles : sk_pairs));
            if (with_workspace) {
                p->dp_tiles = p->num_tiles - sk_tiles;
                p->sk_tiles = sk_tiles;
                p->sk_pairs = sk_pairs;
                p->sk_split = sk_split;
                p->sk_helper_tiles = sk_helper;
                pairs = clusters;
            }
        }
        p->grid = 2 * pairs;
        const int d = cfg.release;
        const int max_slots = max_slots_for_pair(out_dtype, sk, pm);
        int s = cfg.stages > 0 ? cfg.stages : max_slots - d;
        if (s <= d || s + d > max_slots) return GEMM_ERR_CONFIG;
        long long steps_per_cta = (long long)p->k_steps * ceil_div(p->num_tiles, pairs);
        if (p->sk_tiles > 0) steps_per_cta = (long long)p->k_steps * (p->dp_tiles / pairs + 2);
        if (steps_per_cta < s) s = (int)(steps_per_cta > d ? steps_per_cta : d + 1);
        p->stages = s;
        p->release = d;
        p->slots = s + d;
        p->raster_group = cfg.raster_group > 0 ? cfg.raster_group : 8;
        p->tmem_cols = pm == 256 ? 512 : 128;
        p->smem_bytes = smem_request(smem_for_pair(out_dtype, sk, pm, p->slots), p->tmem_cols);
        p->threads = kThreads;
        return GEMM_OK;
    }
    p->cta_group = 1;
    p->dp_tiles = p->num_tiles;
    if (cfg.tile_k != 0 && cfg.tile_k != kBK) return GEMM_ERR_CONFIG;  // deep steps: pairs only

    // Stream-K on single CTAs (stream_k 2, needs a workspace): the iterations
    // of all tiles are dealt out in equal contiguous shares to up to one CTA
    // per SM (at least 16 K steps each), partial tiles meeting through the
    // workspace.  Not a default: on one row of tiles (M = 128, N = K = 8192)
    // it measured 34.5 us where split-K clusters take 28-30 us, because 128
    // SMs already saturate HBM there and a partial parked in global memory
    // costs more than one passed through distributed shared memory.
    if (cfg.split == 0 && cfg.grid == 0 && cfg.stream_k == 2 && p->k_steps > 0) {
        const long long iters = (long long)p->num_tiles * p->k_steps;
        long long ctas = iters / 16;
        if (ctas > num_sms) ctas = num_sms;
        if (ctas > kMaxSkCtas) ctas = kMaxSkCtas;
        if (ctas < 1) ctas = 1;
        p->workspace_bytes = (long long)workspace_for((int)ctas);
        if (with_workspace) {
            p->dp_tiles = 0;
            p->sk_tiles = p->num_tiles;
            p->sk_pairs = (int)ctas;
        }
    }

    int split = cfg.split;
    if (split == 0 && p->sk_tiles > 0) split = 1;
    if (split == 0) {
        split = 1;
        if (p->num_tiles > 0 && 2 * p->num_tiles <= num_sms) {
            split = num_sms / p->num_tiles;
            if (split > kMaxSplit) split = kMaxSplit;
            if (split > p->k_steps / 16) split = p->k_steps / 16;
            // every cluster resident at once (one wave): 48 clusters of three
            // where 46 fit took 32.7 us at 768 x 2048 x 4096, split 2 ~half that
            while (split > 1 && p->num_tiles > fit.clusters[split]) --split;
            if (split < 1) split = 1;
        }
    }
    if (split > 1 && split > p->k_steps) return GEMM_ERR_CONFIG;
    p->split = split;
    if (split > 1) {
        p->grid = p->num_tiles * split;  // one tile per cluster
    } else if (p->sk_tiles > 0) {
        p->grid = p->sk_pairs;
    } else {
        p->grid = p->num_tiles < num_sms ? p->num_tiles : num_sms;
        if (cfg.grid > 0 && cfg.grid < p->grid) p->grid = cfg.grid;
    }
    if (p->grid < 1) p->grid = 1;

    const int d = cfg.release;
    const int max_slots = max_slots_for(tn, out_dtype);
    int s = cfg.stages > 0 ? cfg.stages : max_slots - d;
    if (s <= d) return GEMM_ERR_CONFIG;
    if (s + d > max_slots) return GEMM_ERR_CONFIG;
    const long long ctas_per_tile_slot = split > 1 ? 1 : ceil_div(p->num_tiles, p->grid);
    long long steps_per_cta = (long long)ceil_div(p->k_steps, split) * ctas_per_tile_slot;
    if (p->sk_tiles > 0) steps_per_cta = ((long long)p->sk_tiles * p->k_steps + p->sk_pairs - 1) / p->sk_pairs;
    if (steps_per_cta < s) s = (int)(steps_per_cta > d ? steps_per_cta : d + 1);
    if (split > 1) {
        // partials of other ranks' chunks are parked in (more than two ranks)
        // or pushed into (two ranks, 128 x 256 tiles) the ring: it must hold
        // one fp32 tile
        const int stage_bytes = kBM * kBK * 2 + kBK * tn * 2;
        const int need = (kBM * tn * 4 + stage_bytes - 1) / stage_bytes;
        if (s + d < need) s = need - d;
        if (s + d > max_slots) return GEMM_ERR_CONFIG;
    }
    p->stages = s;
    p->release = d;
    p->slots = s + d;
    p->raster_group = cfg.raster_group > 0 ? cfg.raster_group : 16;
    p->tmem_cols = 2 * tn;
    p->smem_bytes = smem_request(smem_for(tn, out_dtype, p->slots), p->tmem_cols);
    p->threads = kThreads;
    return GEMM_OK;
}

void init_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// 2-D row-major tensor map with a 128-byte swizzle; out-of-range elements
// read as zero and are not written.
int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr, uint64_t inner,
              uint64_t outer, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_TMAP;
}

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0, major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            d.sms = sms;
            d.cc = major * 10 + minor;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return GEMM_OK;
}

template <int OUT, int SK, int PM = kPairBM, int PN = kPairBN, bool PF = false>
int launch_pair(const gemm_plan& plan, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                const KernelParams& kp, cudaStream_t stream, DeviceInfo& dev) {
    auto kern = gemm_f16_pair_kernel<OUT, SK, PM, PN, PF>;
    const int rc = ensure_smem_limit(kern, kSmemLimit, dev.attr_set[PF ? 7 : PM == 128 ? 6 : SK == 128 ? 4 : 3][OUT]);
    if (rc != GEMM_OK) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(plan.grid, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = plan.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&lc, kern, ta, tb, tc, kp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

template <int OUT, int NT>
int launch_small(const gemm_plan& plan, const CUtensorMap& ta, const CUtensorMap& tb, void* C, const KernelParams& kp,
                 cudaStream_t stream, DeviceInfo& dev) {
    auto kern = gemm_f16_small_kernel<OUT, NT>;
    const int rc = ensure_smem_limit(kern, kSmemLimit, dev.attr_set[NT == 8 ? 8 : NT == 16 ? 9 : 10][OUT]);
    if (rc != GEMM_OK) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(plan.grid, 1, 1);
    lc.blockDim = dim3(kSmallThreads, 1, 1);
    lc.dynamicSmemBytes = plan.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, kern, ta, tb, C, kp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

template <int BN, int OUT>
int launch(const gemm_plan& plan, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
           const KernelParams& kp, cudaStream_t stream, DeviceInfo& dev) {
    auto kern = gemm_f16_kernel<BN, OUT>;
    const int rc = ensure_smem_limit(kern, kSmemLimit, dev.attr_set[BN == 64 ? 0 : BN == 128 ? 1 : 2][OUT]);
    if (rc != GEMM_OK) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(plan.grid, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = plan.smem_bytes;
    lc.stream = stream;
    // programmatic serialisation: this kernel's prologue may overlap the tail
    // of the previous kernel in the stream (it waits for that kernel's
    // completion before touching global memory)
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (plan.split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = plan.split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    lc.attrs = attr;
    lc.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&lc, kern, ta, tb, tc, kp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

// CTA-pair clusters the GPU can hold at once (stream-K owners wait on other
// clusters, so every cluster of a launch must be resident together).
int max_pairs_of(DeviceInfo& dev) {
    const int known = dev.max_pairs.load(std::memory_order_acquire);
    if (known > 0) return known;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev.max_pairs.load(std::memory_order_relaxed) == 0) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(dev.sms, 1, 1);
        lc.blockDim = dim3(kThreads, 1, 1);
        lc.dynamicSmemBytes = kSmemLimit;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        auto kern = gemm_f16_pair_kernel<0, 128>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = dev.sms / 2;
        }
        dev.max_pairs.store(n < dev.sms / 2 ? n : dev.sms / 2, std::memory_order_release);
    }
    return dev.max_pairs.load(std::memory_order_relaxed);
}

// Split-K clusters of `size` CTAs the GPU can hold at once (asked once per
// device and size).
int max_clusters_of(DeviceInfo& dev, int size) {
    const int known = dev.max_clusters[size].load(std::memory_order_acquire);
    if (known > 0) return known;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev.max_clusters[size].load(std::memory_order_relaxed) == 0) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((dev.sms / size) * size, 1, 1);
        lc.blockDim = dim3(kThreads, 1, 1);
        lc.dynamicSmemBytes = kSmemLimit;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = size;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        auto kern = gemm_f16_kernel<128, 0>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = fit_estimate(dev.sms).clusters[size];
            if (n < 1) n = 1;
        }
        dev.max_clusters[size].store(n, std::memory_order_release);
    }
    return dev.max_clusters[size].load(std::memory_order_relaxed);
}

Fit fit_of(DeviceInfo& dev) {
    Fit f;
    f.clusters[0] = 0;
    f.clusters[1] = dev.sms;
    f.clusters[2] = max_pairs_of(dev);
    for (int c = 3; c <= kMaxSplit; ++c) f.clusters[c] = max_clusters_of(dev, c);
    return f;
}

gemm_config current_config() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_cfg;
}

#ifdef TCGEMM_TRACE
// The trace build's buffer (gemm_f16_trace_buffer) and its launch count.
struct TraceState {
    unsigned long long* buf = nullptr;
    int slots = 0, ctas = 0, events = 0;
    unsigned long long launches = 0;
};
TraceState g_trace;
std::mutex g_trace_mu;

// Where this launch records (NULL: not traced), advancing the launch count.
unsigned long long* next_trace_slot(int* ctas, int* events) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace.buf) return nullptr;
    const unsigned long long slot = g_trace.launches++ % (unsigned long long)g_trace.slots;
    *ctas = g_trace.ctas;
    *events = g_trace.events;
    return g_trace.buf + slot * (unsigned long long)g_trace.ctas * kTraceRoles * g_trace.events * 2;
}
#endif

// Encode the tensor maps and launch one planned problem (arguments already
// checked; `plan` made with `cfg` for this device; the workspace, if the plan
// uses one, large enough).
int launch_planned(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K, int out_dtype,
                   void* workspace, gemm_stream_t stream, bool accumulate, const gemm_config& cfg,
                   const gemm_plan& plan, DeviceInfo* dev) {
    int rc = GEMM_OK;
    std::call_once(g_encode_once, init_encode);
    if (!g_encode) return GEMM_ERR_CUDA;
    CUtensorMap ta, tb, tc;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (K > 0) {
        // each CTA loads its rows of the tile: 128, or 64 on a 128 x 128 pair tile
        rc = encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, (uint64_t)K, (uint64_t)M, kBK,
                       (uint32_t)(plan.tile_m / plan.cta_group));
        if (rc != GEMM_OK) return rc;
        rc = encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B, (uint64_t)N, (uint64_t)K, 64, plan.tile_k);
        if (rc != GEMM_OK) return rc;
    }
    if (out_dtype == GEMM_OUT_F16)
        rc = encode_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, C, (uint64_t)N, (uint64_t)M, 64, 32);
    else
        rc = encode_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, (uint64_t)N, (uint64_t)M, 32, 32);
    if (rc != GEMM_OK) return rc;

    KernelParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.M = M;
    kp.N = N;
    kp.K = K;
    kp.tiles_m = plan.tiles_m;
    kp.tiles_n = plan.tiles_n;
    kp.k_blocks = plan.k_steps;
    kp.raster_group = plan.raster_group;
    kp.slots = plan.slots;
    kp.release = plan.release;
    kp.split = plan.split;
    kp.wait_limit = cfg.wait_limit > 0 ? cfg.wait_limit : kDefaultWaitLimit;
    kp.inject = cfg.inject_stall;
    kp.dp_tiles = plan.dp_tiles;
    kp.sk_tiles = plan.sk_tiles;
    kp.sk_pairs = plan.sk_pairs;
    kp.sk_split = plan.sk_split;
    kp.sk_helper_tiles = plan.sk_helper_tiles;
    kp.c_in = accumulate ? C : nullptr;
    // a small pair launch (one unit per pair, at most half the SMs) starts while
    // the previous kernel runs: its CTAs prefetch their operands into L2 first
    // (256^3: 3.55 -> 3.27 us, 512^3: 4.56 -> 4.30 us in CUDA graphs)
    const bool prefetch = plan.cta_group == 2 && plan.tile_m == 128 && plan.sk_tiles == 0 && plan.k_steps > 0 &&
                          plan.num_tiles <= plan.grid / 2 && 2 * plan.grid <= dev->sms;
    if (prefetch) kp.pf_steps = plan.k_steps < kPrefetchSteps ? plan.k_steps : kPrefetchSteps;
#ifdef TCGEMM_TRACE
    kp.trace = next_trace_slot(&kp.trace_ctas, &kp.trace_events);
#endif
    if (plan.sk_tiles > 0) {
        // flags first, then the partial tiles (layout of workspace_for)
        unsigned e = ++g_epoch;
        if (e == 0) e = ++g_epoch;  // 0 is what a fresh (zero-filled) workspace holds
        kp.epoch = e;
        kp.flags = reinterpret_cast<unsigned*>(workspace);
        kp.ws = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + kFlagBytes);
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan.cta_group == 1 && plan.tile_m < kBM) {
        if (out_dtype == GEMM_OUT_F16)
            return plan.tile_m == 8 ? launch_small<0, 8>(plan, ta, tb, C, kp, s, *dev)
                   : plan.tile_m == 16 ? launch_small<0, 16>(plan, ta, tb, C, kp, s, *dev)
                                       : launch_small<0, 32>(plan, ta, tb, C, kp, s, *dev);
        return plan.tile_m == 8 ? launch_small<1, 8>(plan, ta, tb, C, kp, s, *dev)
               : plan.tile_m == 16 ? launch_small<1, 16>(plan, ta, tb, C, kp, s, *dev)
                                   : launch_small<1, 32>(plan, ta, tb, C, kp, s, *dev);
    }
    if (prefetch)
        return out_dtype == GEMM_OUT_F16 ? launch_pair<0, 128, 128, 128, true>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch_pair<1, 128, 128, 128, true>(plan, ta, tb, tc, kp, s, *dev);
    if (plan.cta_group == 2 && plan.tile_m == 128)
        return out_dtype == GEMM_OUT_F16 ? launch_pair<0, 128, 128, 128>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch_pair<1, 128, 128, 128>(plan, ta, tb, tc, kp, s, *dev);
    if (plan.cta_group == 2 && plan.tile_k == 128)
        return out_dtype == GEMM_OUT_F16 ? launch_pair<0, 128>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch_pair<1, 128>(plan, ta, tb, tc, kp, s, *dev);
    if (plan.cta_group == 2)
        return out_dtype == GEMM_OUT_F16 ? launch_pair<0, 64>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch_pair<1, 64>(plan, ta, tb, tc, kp, s, *dev);
    if (plan.tile_n == 256)
        return out_dtype == GEMM_OUT_F16 ? launch<256, 0>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch<256, 1>(plan, ta, tb, tc, kp, s, *dev);
    if (plan.tile_n == 64)
        return out_dtype == GEMM_OUT_F16 ? launch<64, 0>(plan, ta, tb, tc, kp, s, *dev)
                                         : launch<64, 1>(plan, ta, tb, tc, kp, s, *dev);
    return out_dtype == GEMM_OUT_F16 ? launch<128, 0>(plan, ta, tb, tc, kp, s, *dev)
                                     : launch<128, 1>(plan, ta, tb, tc, kp, s, *dev);
}

int run(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K, int out_dtype, void* workspace,
        size_t workspace_bytes, gemm_stream_t stream, bool accumulate = false) {
    int rc = check_args(A, B, C, M, N, K, out_dtype, true);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    if (workspace && ((uintptr_t)workspace & 255)) return GEMM_ERR_ALIGN;
    const gemm_config cfg = current_config();
    DeviceInfo* dev = nullptr;
    rc = device_info(&dev);
    if (rc != GEMM_OK) return rc;
    if (dev->cc != 103) return GEMM_ERR_ARCH;
    gemm_plan plan;
    rc = plan_impl(M, N, K, out_dtype, dev->sms, fit_of(*dev), workspace != nullptr, cfg, &plan);
    if (rc != GEMM_OK) return rc;
    if (plan.sk_tiles > 0 && (size_t)plan.workspace_bytes > workspace_bytes) return GEMM_ERR_WORKSPACE;
    return launch_planned(A, B, C, M, N, K, out_dtype, workspace, stream, accumulate, cfg, plan, dev);
}

int plan_entry(int M, int N, int K, int out_dtype, int num_sms, bool with_workspace, gemm_plan* out) {
    if (!out) return GEMM_ERR_NULL;
    int rc = check_args(nullptr, nullptr, nullptr, M, N, K, out_dtype, false);
    if (rc < 0) return rc;
    if (num_sms < 0) return GEMM_ERR_DIM;
    if (num_sms == 0) {
        DeviceInfo* dev = nullptr;
        rc = device_info(&dev);
        if (rc != GEMM_OK) return rc;
        return plan_impl(M, N, K, out_dtype, dev->sms, fit_of(*dev), with_workspace, current_config(), out);
    }
    return plan_impl(M, N, K, out_dtype, num_sms, fit_estimate(num_sms), with_workspace, current_config(), out);
}

}  // namespace

extern "C" {

int gemm_f16(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K, int out_dtype,
             gemm_stream_t stream) {
    return run(A, B, C, M, N, K, out_dtype, nullptr, 0, stream);
}

int gemm_f16_ws(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K, int out_dtype,
                void* workspace, size_t workspace_bytes, gemm_stream_t stream) {
    return run(A, B, C, M, N, K, out_dtype, workspace, workspace_bytes, stream);
}

int gemm_f16_acc(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K, int out_dtype,
                 gemm_stream_t stream) {
    return run(A, B, C, M, N, K, out_dtype, nullptr, 0, stream, true);
}

int gemm_f16_plan(int M, int N, int K, int out_dtype, int num_sms, gemm_plan* out) {
    return plan_entry(M, N, K, out_dtype, num_sms, false, out);
}

int gemm_f16_plan_ws(int M, int N, int K, int out_dtype, int num_sms, gemm_plan* out) {
    return plan_entry(M, N, K, out_dtype, num_sms, true, out);
}

int gemm_f16_workspace_size(int M, int N, int K, int out_dtype, int num_sms, size_t* bytes) {
    if (!bytes) return GEMM_ERR_NULL;
    *bytes = 0;
    gemm_plan plan;
    int rc = plan_entry(M, N, K, out_dtype, num_sms, true, &plan);
    if (rc != GEMM_OK) return rc;
    *bytes = plan.sk_tiles > 0 ? (size_t)plan.workspace_bytes : 0;
    return GEMM_OK;
}

int gemm_f16_set_config(const gemm_config* cfg) {
    gemm_config c = {};
    if (cfg) c = *cfg;
    int rc = check_config(c);
    if (rc != GEMM_OK) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    g_cfg = c;
    return GEMM_OK;
}

int gemm_f16_get_config(gemm_config* out) {
    if (!out) return GEMM_ERR_NULL;
    std::lock_guard<std::mutex> lk(g_mu);
    *out = g_cfg;
    return GEMM_OK;
}

const char* gemm_f16_strerror(int code) {
    switch (code) {
        case GEMM_OK: return "success";
        case GEMM_ERR_NULL: return "a required pointer is NULL";
        case GEMM_ERR_DIM: return "M, N or K is negative or the problem is too large to index";
        case GEMM_ERR_DTYPE: return "out_dtype must be GEMM_OUT_F16 (0) or GEMM_OUT_F32 (1)";
        case GEMM_ERR_ALIGN: return "pointers must be 16-byte aligned and N, K multiples of 8";
        case GEMM_ERR_ALIAS: return "C overlaps A or B";
        case GEMM_ERR_CONFIG: return "invalid tuning config for this problem (stages must exceed release; tile_n 64, 128 or 256; ring must fit shared memory; split and CTA pairs need K steps)";
        case GEMM_ERR_TMAP: return "the driver refused a TMA tensor-map encoding";
        case GEMM_ERR_LAUNCH: return "kernel launch failed";
        case GEMM_ERR_CUDA: return "no usable CUDA device or driver";
        case GEMM_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
        case GEMM_ERR_DEVICE_TIMEOUT: return "a kernel's bounded device-side wait ran out";
        case GEMM_ERR_WORKSPACE: return "the workspace is smaller than gemm_f16_workspace_size reports";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "the problem needs more stream-K scratch than gemm_f16_noalloc's fixed array holds (160 CTAs' partial tiles)";
        default: return "unknown gemm_status code";
    }
}

int gemm_f16_device_status(int* site, int reset) {
    if (site) *site = 0;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != GEMM_OK) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (reset && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    }
    if (site) *site = (int)v;
    return v == 0 ? GEMM_OK : GEMM_ERR_DEVICE_TIMEOUT;
}

int gemm_f16_abi_version(void) { return 2; }

}  // extern "C"

#ifdef TCGEMM_CHECK
namespace {

// Every access a launch of plan `p` makes, at the granularity the kernels
// test them (bounds.cuh): ring slots and their barriers, staging buffers,
// accumulators, split-K blocks, workspace slots.  Returns the first failing
// site, 0 if none.  L: the kernel's layout; pair: the CTA-pair kernel.
template <class L, bool kPair>
unsigned check_layout(const gemm_plan& p, int acc_cols, int out_cols) {
    const int S = p.slots;
    if (S < 1 || S > kMaxStages) return kSiteSmemBounds;  // full[] and empty[] hold kMaxStages
    const Carve cv = carve(S, L::kABytes, L::kBBytes, L::kStagingBytes, L::kNumBars);
    // the carve-up, after the worst alignment skip, within the shared memory requested
    if (cv.end + kMaxAlignSkip > (uint32_t)p.smem_bytes) return kSiteSmemBounds;
    const uint32_t ring_a = (uint32_t)S * L::kABytes, ring_b = (uint32_t)S * L::kBBytes;
    const uint32_t staging_all = 4u * 2u * L::kStagingBytes, bars = (uint32_t)L::kNumBars * 8u;
    for (int st = 0; st < S; ++st) {
        const int rs = (st - p.release + S) % S;
        if (!(holds(cv.bar, bars, cv.bar + 8u * st, 8) && holds(cv.bar, bars, cv.bar + 8u * (kMaxStages + st), 8) &&
              holds(cv.bar, bars, cv.bar + 8u * (kMaxStages + rs), 8) &&
              holds(cv.a, ring_a, cv.a + st * L::kABytes, L::kABytes) &&
              holds(cv.b, ring_b, cv.b + st * L::kBBytes, L::kBBytes)))
            return kSiteSmemBounds;
    }
    for (int q = 0; q < 4; ++q)
        if (!holds(cv.c, staging_all, cv.c + (uint32_t)(q * 2 * L::kStagingBytes), 2 * L::kStagingBytes))
            return kSiteSmemBounds;
    // Tensor Memory: an allocation is a power of two from 32 to 512 columns,
    // the one the plan reports, and holds both accumulators
    const int tc = L::kTmemCols;
    if (tc < 32 || tc > 512 || (tc & (tc - 1)) || tc != p.tmem_cols || 2 * acc_cols > tc) return kSiteTmemBounds;
    if (!kPair && p.split > 1) {
        const int chunks = p.tile_n / out_cols;
        const uint32_t block = (uint32_t)(out_cols / 4 * 32 * 16);
        const bool to_staging = (chunks + 1) / 2 * block <= 2u * L::kStagingBytes;
        for (int c = 0; c < chunks; ++c)
            for (int q = 0; q < 4; ++q) {
                const bool ok = p.split == 2 && to_staging
                                    ? holds(cv.c, staging_all, cv.c + push_offset(c, q, block, L::kStagingBytes), block)
                                    : holds(cv.a, ring_a + ring_b, cv.a + park_offset(c, q, block), block);
                if (!ok) return kSiteSmemBounds;
            }
    }
    if (p.sk_tiles > 0) {
        // partial slots: one per sharing cluster, or one per shared tile under helpers
        const long long ctas = (long long)(p.sk_split > 0 ? p.sk_tiles : p.sk_pairs) * (kPair ? 2 : 1);
        if (p.sk_split > 0 && (!kPair || p.sk_split >= p.k_steps || p.sk_helper_tiles < 1 ||
                               (long long)(p.sk_pairs - p.sk_tiles) * p.sk_helper_tiles < p.sk_tiles))
            return kSiteWorkspaceBounds;  // helpers that leave a shared tile without its rest
        if (ctas > kMaxSkCtas || (size_t)p.workspace_bytes < workspace_for((int)ctas)) return kSiteWorkspaceBounds;
        // a partial of up to 128 x (accumulator columns x lanes folded) fp32 per CTA
        if ((long long)kBM * acc_cols > kPartialFloats) return kSiteWorkspaceBounds;
    }
    return 0;
}

}  // namespace

// The small kernel's carve-up (K blocks, the C tile, the barriers) inside the
// shared memory the plan asks for, its K blocks within the kernel's limit,
// one tile per CTA and its 32 TMEM columns.
template <class L>
unsigned check_small(const gemm_plan& p) {
    if (p.k_steps < 1 || p.k_steps > kSmallMaxKB || p.grid != p.num_tiles || p.split != 1) return kSiteSmemBounds;
    const long long need = 1023 + (long long)p.k_steps * L::kBlockBytes + L::kStageBytes + (kSmallMaxKB + 1) * 8 + 8;
    if (need > p.smem_bytes || p.smem_bytes > kSmemLimit) return kSiteSmemBounds;
    if (p.tmem_cols != L::kTmemCols) return kSiteTmemBounds;
    return 0;
}

extern "C" int gemm_f16_check_plan(const gemm_plan* plan, int out_dtype, int* site) {
    if (!plan || !site) return GEMM_ERR_NULL;
    *site = 0;
    if (out_dtype != GEMM_OUT_F16 && out_dtype != GEMM_OUT_F32) return GEMM_ERR_DTYPE;
    const gemm_plan& p = *plan;
    const bool f16 = out_dtype == GEMM_OUT_F16;
    unsigned s = kSiteSmemBounds;  // a plan no kernel runs
    if (p.cta_group == 2 && p.tile_m == 128 && p.tile_n == 128 && p.tile_k == 128)
        s = f16 ? check_layout<PairLayout<0, 128, 128, 128>, true>(p, 64, 64)
                : check_layout<PairLayout<1, 128, 128, 128>, true>(p, 64, 32);
    else if (p.cta_group == 2 && p.tile_m == 256 && p.tile_n == 256 && p.tile_k == 128)
        s = f16 ? check_layout<PairLayout<0, 128>, true>(p, 256, 64) : check_layout<PairLayout<1, 128>, true>(p, 256, 32);
    else if (p.cta_group == 2 && p.tile_m == 256 && p.tile_n == 256 && p.tile_k == 64)
        s = f16 ? check_layout<PairLayout<0, 64>, true>(p, 256, 64) : check_layout<PairLayout<1, 64>, true>(p, 256, 32);
    else if (p.cta_group == 1 && p.tile_m == 128 && p.tile_k == 64 && p.tile_n == 256)
        s = f16 ? check_layout<Layout<256, 0>, false>(p, 256, 64) : check_layout<Layout<256, 1>, false>(p, 256, 32);
    else if (p.cta_group == 1 && p.tile_m == 128 && p.tile_k == 64 && p.tile_n == 128)
        s = f16 ? check_layout<Layout<128, 0>, false>(p, 128, 64) : check_layout<Layout<128, 1>, false>(p, 128, 32);
    else if (p.cta_group == 1 && p.tile_m == 128 && p.tile_k == 64 && p.tile_n == 64)
        s = f16 ? check_layout<Layout<64, 0>, false>(p, 64, 64) : check_layout<Layout<64, 1>, false>(p, 64, 32);
    else if (p.cta_group == 1 && p.tile_n == kSmallBN && p.tile_k == 64 && p.tile_m == 8)
        s = f16 ? check_small<SmallLayout<0, 8>>(p) : check_small<SmallLayout<1, 8>>(p);
    else if (p.cta_group == 1 && p.tile_n == kSmallBN && p.tile_k == 64 && p.tile_m == 16)
        s = f16 ? check_small<SmallLayout<0, 16>>(p) : check_small<SmallLayout<1, 16>>(p);
    else if (p.cta_group == 1 && p.tile_n == kSmallBN && p.tile_k == 64 && p.tile_m == 32)
        s = f16 ? check_small<SmallLayout<0, 32>>(p) : check_small<SmallLayout<1, 32>>(p);
    *site = (int)s;
    return s == 0 ? GEMM_OK : GEMM_ERR_CONFIG;
}
#endif

extern "C" {

#ifdef TCGEMM_TRACE
int gemm_f16_trace_buffer(void* buffer, size_t bytes, int launch_slots, int ctas, int events) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!buffer) {
        g_trace = TraceState();
        return GEMM_OK;
    }
    if (launch_slots < 1 || ctas < 1 || events < 1) return GEMM_ERR_NULL;
    if ((uintptr_t)buffer & 7) return GEMM_ERR_ALIGN;
    const unsigned long long need = (unsigned long long)launch_slots * ctas * kTraceRoles * events * 16ull;
    if (bytes < need) return GEMM_ERR_NULL;
    g_trace.buf = static_cast<unsigned long long*>(buffer);
    g_trace.slots = launch_slots;
    g_trace.ctas = ctas;
    g_trace.events = events;
    g_trace.launches = 0;
    return GEMM_OK;
}
#endif

int add_matrices_f32(const float* X, const float* Y, float* Z, int M, int N, gemm_stream_t stream) {
    if (M < 0 || N < 0) return GEMM_ERR_DIM;
    if (N % 4 != 0) return GEMM_ERR_ALIGN;
    if ((long long)ceil_div(M, kAddBM) * ceil_div(N, kAddBN) > INT_MAX) return GEMM_ERR_DIM;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!X || !Y || !Z) return GEMM_ERR_NULL;
    const uintptr_t x = (uintptr_t)X, y = (uintptr_t)Y, z = (uintptr_t)Z;
    if ((x | y | z) & 15) return GEMM_ERR_ALIGN;
    // Z may be X or Y itself (every element is read before it is written), but
    // may not partly overlap either
    const uint64_t bytes = (uint64_t)M * N * 4;
    if (z != x && z < x + bytes && x < z + bytes) return GEMM_ERR_ALIAS;
    if (z != y && z < y + bytes && y < z + bytes) return GEMM_ERR_ALIAS;
    const gemm_config cfg = current_config();
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != GEMM_OK) return rc;
    if (dev->cc != 103) return GEMM_ERR_ARCH;
    std::call_once(g_encode_once, init_encode);
    if (!g_encode) return GEMM_ERR_CUDA;
    CUtensorMap tx, ty, tz;
    rc = encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, X, (uint64_t)N, (uint64_t)M, kAddBN, kAddBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != GEMM_OK) return rc;
    rc = encode_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Y, (uint64_t)N, (uint64_t)M, kAddBN, kAddBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != GEMM_OK) return rc;
    rc = encode_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Z, (uint64_t)N, (uint64_t)M, kAddBN,
                   kAddBM / kAddWarps, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != GEMM_OK) return rc;
    AddParams ap;
    ap.M = M;
    ap.N = N;
    ap.tiles_m = ceil_div(M, kAddBM);
    ap.tiles_n = ceil_div(N, kAddBN);
    ap.slots = 3;  // at least 2: a slot is freed only after the next tile's store
    ap.wait_limit = cfg.wait_limit > 0 ? cfg.wait_limit : kDefaultWaitLimit;
    const int tiles = ap.tiles_m * ap.tiles_n;
    const int smem = AddLayout::smem_bytes(ap.slots);
    rc = ensure_smem_limit(add_f32_kernel, smem, dev->attr_set[5][0]);
    if (rc != GEMM_OK) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(tiles < dev->sms ? tiles : dev->sms, 1, 1);
    lc.blockDim = dim3(kAddThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, add_f32_kernel, tx, ty, tz, ap) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // extern "C"

// ---- stream-K without any allocation ---------------------------------------------
//
// For callers that cannot allocate device memory at the point of the call:
// allocators or runtimes that must not re-enter the CUDA allocator; plugins
// that are handed only their input and output buffers; latency-critical code
// where cudaMalloc may synchronise the device.  gemm_f16_noalloc runs
// the same plan as gemm_f16_ws, with the stream-K scratch (flags and fp32
// partial tiles) in one fixed array in device memory instead of a workspace
// the caller passes in.

namespace {

// The scratch: room for the flags and the partial tiles of kNoAllocMaxCtas
// CTAs (80 CTA pairs, more than a 152-SM GB300 ever shares), held in every
// GPU that loads this library until the process exits.  Zero at module load.
// Calls share it and it keeps what the last call wrote.  A flag word only
// ever holds 0 or some launch's epoch (the flag area has one fixed size, so
// no plan keeps a partial tile there), and an epoch never repeats from one
// launch to the next; an owner zeroes each flag it has consumed.
constexpr int kNoAllocMaxCtas = 160;
constexpr size_t kNoAllocScratchBytes = workspace_for(kNoAllocMaxCtas);  // 20 MiB + 16 KiB
static_assert(kNoAllocScratchBytes == (20u << 20) + kFlagBytes, "scratch size as documented");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  The array's name in
// host code is only a host-side handle, so the address is asked of the runtime
// once per device (with that device current) and then reused.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" int gemm_f16_noalloc(const gemm_f16_t* A, const gemm_f16_t* B, void* C, int M, int N, int K,
                                int out_dtype, gemm_stream_t stream) {
    int rc = check_args(A, B, C, M, N, K, out_dtype, true);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    // one read of the config and one plan serve both the size check and the launch
    const gemm_config cfg = current_config();
    DeviceInfo* dev = nullptr;
    rc = device_info(&dev);
    if (rc != GEMM_OK) return rc;
    if (dev->cc != 103) return GEMM_ERR_ARCH;
    gemm_plan plan;
    rc = plan_impl(M, N, K, out_dtype, dev->sms, fit_of(*dev), true, cfg, &plan);
    if (rc != GEMM_OK) return rc;
    if (plan.sk_tiles > 0 && (size_t)plan.workspace_bytes > kNoAllocScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;
    // looked up on every call (cached after the first on this device), whether
    // or not this plan shares tiles, so the first call does the set-up
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != GEMM_OK) return rc;
    return launch_planned(A, B, C, M, N, K, out_dtype, plan.sk_tiles > 0 ? scratch : nullptr, stream, false, cfg,
                          plan, dev);
}
