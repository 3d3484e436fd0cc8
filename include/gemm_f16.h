/*
 * gemm_f16.h - C ABI of the GB300 (sm_103a) pipelined tiled fp16 GEMM.
 *
 * The operation is the matmul of "Quickstart: GPU" (Pallas Mosaic GPU),
 * section "Pipelining: a matmul kernel": matmul(a, b, out_dtype)
 * with m, k = a.shape and _, n = b.shape, fp16 operands, an fp32 Tensor Core
 * accumulator (plgpu.ACC) and a final conversion acc.astype(out_dtype):
 *
 *     C[i][j] = out_dtype( sum_k  A[i][k] * B[k][j] ),  accumulated in fp32.
 *
 * The parallel grid of output tiles, the sequential pipeline along K and its
 * two knobs (max_concurrent_steps, delay_release) come from the same page,
 * from "JAX Pallas Mosaic GPU 快速上手" (section "深入emit_pipeline的关键参数")
 * and from "JAX Pallas 软件流水线 Software Pipelining 完全指南" (sections 3,
 * 4 and 9.2).  Here they are realised with TMA,
 * an mbarrier-guarded shared-memory ring, tcgen05.mma into Tensor Memory and
 * a persistent tile scheduler.
 *
 * Conventions for every entry point:
 *   - Matrices are dense and row-major: A is M x K (row stride K elements),
 *     B is K x N (row stride N), C is M x N (row stride N).
 *   - A, B and C are DEVICE pointers owned by the caller.  The library never
 *     allocates, frees or synchronises them; it keeps only a small per-device
 *     cache (SM count, kernel attributes) and one process-wide tuning config.
 *   - Every entry point may be called from several host threads at once; the
 *     cache is filled under a lock on first use.
 *   - Return value: 0 on success, a negative gemm_status code otherwise.
 *     Argument checks run on the host before any CUDA call; no exceptions are
 *     thrown and nothing is printed.
 */
#ifndef TCGEMM_GEMM_F16_H
#define TCGEMM_GEMM_F16_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One IEEE 754 binary16 value as stored in memory (same layout as CUDA's
 * __half; pass a __half* with a cast). */
typedef unsigned short gemm_f16_t;

/* The same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OUT_F16 = 0, /* C is fp16, rounded to nearest even from the fp32 accumulator */
    GEMM_OUT_F32 = 1  /* C is the fp32 accumulator */
} gemm_out_dtype;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_NULL = -1,           /* a required pointer is NULL */
    GEMM_ERR_DIM = -2,            /* M, N or K negative, or the problem too large to index */
    GEMM_ERR_DTYPE = -3,          /* out_dtype not a gemm_out_dtype */
    GEMM_ERR_ALIGN = -4,          /* a pointer not 16-byte aligned, or N or K not a multiple of 8
                                     (TMA needs 16-byte-aligned rows) */
    GEMM_ERR_ALIAS = -5,          /* C overlaps A or B (inputs are read-only, the output write-only) */
    GEMM_ERR_CONFIG = -6,         /* invalid tuning config, e.g. release >= stages */
    GEMM_ERR_TMAP = -7,           /* the driver refused a tensor-map encoding */
    GEMM_ERR_LAUNCH = -8,         /* the kernel launch failed */
    GEMM_ERR_CUDA = -9,           /* no usable CUDA device or driver entry point */
    GEMM_ERR_ARCH = -10,          /* the current device is not compute capability 10.3 */
    GEMM_ERR_DEVICE_TIMEOUT = -11, /* a kernel's bounded wait ran out (see gemm_f16_device_status) */
    GEMM_ERR_WORKSPACE = -12,      /* the workspace given to gemm_f16_ws is smaller than its plan needs */
    GEMM_ERR_SCRATCH_LIMIT = -13   /* the problem needs more scratch than gemm_f16_noalloc's fixed array */
} gemm_status;

/* What the planner chose for one problem (gemm_f16_plan). */
typedef struct {
    int cta_group;              /* 1: one CTA per tile; 2: a CTA pair (two SMs) per tile,
                                   256 x 256 or 128 x 128 */
    int tile_m, tile_n, tile_k; /* output tile and K step (elements); tile_m 8, 16 or 32 with
                                   tile_n 64 (cta_group 1, 128 threads): the small-problem kernel,
                                   one wave of CTAs holding all of K (at most 512) at once */
    int tiles_m, tiles_n;       /* ceil(M/tile_m), ceil(N/tile_n) */
    int num_tiles;              /* tiles_m * tiles_n: one owner CTA each */
    int k_steps;                /* ceil(K/tile_k): the sequential pipeline length */
    int stages;                 /* loads in flight ahead of the MMA (max_concurrent_steps) */
    int release;                /* extra steps before a buffer is reused (delay_release) */
    int slots;                  /* shared-memory ring buffers: stages + release */
    int split;                  /* CTAs (one thread-block cluster) sharing each tile along K */
    int grid;                   /* CTAs launched: persistent, num_tiles * split with split-K, or
                                   num_tiles (the small kernel) */
    int raster_group;           /* m-blocks per raster group */
    int smem_bytes;             /* dynamic shared memory per CTA */
    int tmem_cols;              /* Tensor Memory columns per CTA */
    int threads;                /* threads per CTA */
    int dp_tiles;               /* tiles run data-parallel (all of them without stream-K) */
    int sk_tiles;               /* tiles whose K iterations are shared by clusters (stream-K) */
    int sk_pairs;               /* clusters sharing them: CTA pairs, or single CTAs (cta_group 1) */
    long long workspace_bytes;  /* workspace gemm_f16_ws needs for its stream-K plan; 0 if none */
    int sk_split;               /* 0: the shared K iterations are dealt out in even contiguous shares;
                                   > 0 (CTA pairs, a last wave more than half full): pair i runs K steps
                                   [0, sk_split) of shared tile dp_tiles + i, and the pairs idle in that
                                   wave ("helpers") run steps [sk_split, k_steps) of the shared tiles, one
                                   after another; the data-parallel tiles follow on every pair */
    int sk_helper_tiles;        /* with sk_split > 0: shared tiles each helper pair runs */
} gemm_plan;

/* Tuning override.  Zero in a field means "planner default". */
typedef struct {
    int tile_n;            /* 0, 64, 128 or 256 */
    int stages;            /* 0 or 1..8: loads in flight (max_concurrent_steps) */
    int release;           /* 0..7: delay_release; stages must exceed it, and
                              stages + release buffers must fit shared memory */
    int grid;              /* 0 = min(num_tiles, SM count); else a cap on the CTAs launched */
    int raster_group;      /* 0 or >= 1 */
    long long wait_limit;  /* 0 = about one second; else clock cycles one device wait may take */
    int split;             /* 0 = planner default; 1 = no split-K; 2..8 = CTAs per tile along K */
    int cta_group;         /* 0 = planner default; 1 = one CTA per tile; 2 = CTA pairs, no
                              split: 256 x 256 tiles (tile_n 0 or 256; 128 rows per SM)
                              or 128 x 128 tiles (tile_n 128; 64 rows per SM) */
    int tile_k;            /* 0 = planner default; K depth of one pipeline step: 64, or 128
                              (CTA pairs only; 128 x 128 pair tiles take 128 only) */
    int stream_k;          /* 0 = planner default (gemm_f16_ws shares the last, partly
                              filled wave of CTA-pair tiles); 1 = never; 2 = share the K
                              iterations of every tile, also on single CTAs (needs a
                              workspace) */
    int inject_stall;      /* test hook: 1 makes every CTA's producer issue no loads, so
                              the MMA warp's bounded wait runs out and the kernel reports
                              GEMM_ERR_DEVICE_TIMEOUT instead of finishing.  0 in normal use. */
} gemm_config;

/*
 * C = A * B (fp16 x fp16, fp32 accumulation), written as out_dtype.
 *
 *   A          device, M x K fp16, row-major, 16-byte aligned, read-only
 *   B          device, K x N fp16, row-major, 16-byte aligned, read-only
 *   C          device, M x N of out_dtype, row-major, 16-byte aligned; must not
 *              overlap A or B; every element is written
 *   M, N, K    >= 0; N and K multiples of 8 (16-byte rows for TMA).  M, N and K
 *              need not be multiples of the tile: edge tiles are zero-filled on
 *              load and clipped on store.  M == 0 or N == 0 is a no-op; K == 0
 *              writes zeros (the empty sum).
 *   out_dtype  GEMM_OUT_F16 or GEMM_OUT_F32
 *   stream     CUDA stream the kernel is enqueued on; the call is asynchronous
 *              and C is valid once the stream reaches this point
 *
 * Pointers may be NULL only where nothing is read or written through them
 * (A and B when K == 0; all three when M == 0 or N == 0).  All three must
 * point into memory of the current device: the call does not ask the driver
 * where a pointer points, so host memory or another device's memory is not
 * detected here (the Python binding checks its tensors).
 * Errors: GEMM_ERR_DTYPE, GEMM_ERR_DIM, GEMM_ERR_NULL, GEMM_ERR_ALIGN,
 * GEMM_ERR_ALIAS, GEMM_ERR_CONFIG before any CUDA call; GEMM_ERR_CUDA,
 * GEMM_ERR_ARCH, GEMM_ERR_TMAP, GEMM_ERR_LAUNCH after.  A device-side timeout
 * is not seen here (the launch is asynchronous): read gemm_f16_device_status.
 */
int gemm_f16(const gemm_f16_t *A, const gemm_f16_t *B, void *C, int M, int N, int K, int out_dtype,
             gemm_stream_t stream);

/*
 * C += A * B: the product accumulated into the values C already holds
 * (in fp32, then rounded once to out_dtype).  This is the reduction of the
 * "JAX Pallas 软件流水线 Software Pipelining 完全指南", section 7.2 (a sum
 * accumulated into the output block along the innermost grid axis), started
 * from C instead of zero, C being both an input and the output as section 7.1
 * allows for aliased buffers.  C is read and written; it must still not
 * overlap A or B.  K == 0 leaves C as it was.  Arguments and errors as
 * gemm_f16.
 */
int gemm_f16_acc(const gemm_f16_t *A, const gemm_f16_t *B, void *C, int M, int N, int K, int out_dtype,
                 gemm_stream_t stream);

/*
 * As gemm_f16, with a caller-owned device workspace for stream-K.  When the
 * tiles of the CTA-pair kernel do not fill the last wave, the K iterations of
 * that wave's tiles are shared evenly by the pairs, whose partial tiles meet
 * through the workspace.  `workspace_bytes` must be at least what
 * gemm_f16_workspace_size reports, else GEMM_ERR_WORKSPACE.
 *
 *   workspace  device pointer, 256-byte aligned; zero-filled by the caller
 *              before its FIRST use with this library (the library keeps it
 *              valid for later calls); NULL runs exactly as gemm_f16
 *   layout     16 KiB of flags (one 32-bit word per epilogue warp of up to
 *              1024 CTAs), then one 128 x 256 fp32 partial tile (128 KiB) per
 *              CTA that shares tiles.  A flag holds 0 or the value of the
 *              launch whose partial is ready; the warp that consumes a
 *              partial sets its flag back to 0, so a launch captured in a
 *              CUDA graph and replayed waits for each replay's own partials.
 *   ownership  the caller's; it may be reused by the next call on the same
 *              stream, but two calls that may overlap on the GPU must not
 *              share one workspace.  After a launch that reported
 *              GEMM_ERR_DEVICE_TIMEOUT, zero it again before reuse.
 * Errors: those of gemm_f16, GEMM_ERR_ALIGN for a misaligned workspace and
 * GEMM_ERR_WORKSPACE for a short one.
 */
int gemm_f16_ws(const gemm_f16_t *A, const gemm_f16_t *B, void *C, int M, int N, int K, int out_dtype,
                void *workspace, size_t workspace_bytes, gemm_stream_t stream);

/*
 * As gemm_f16_ws, for callers that cannot allocate device memory when they
 * call: a memory allocator or runtime that must not re-enter the CUDA
 * allocator from inside its own calls; a plugin or operator that its host
 * framework hands only input and output buffers, with no allocation hook; code
 * on a latency-critical path, where cudaMalloc may synchronise the device.
 * The pages have no counterpart; this is an interface convenience of this
 * library.
 *
 * The stream-K scratch lives in one fixed array of 20 MiB + 16 KiB in device
 * memory (the 16 KiB of flags and the 128 KiB partial tiles of at most 160
 * CTAs, i.e. 80 CTA pairs), which every GPU that loads this library holds
 * until the process exits.  Nothing is allocated or freed by the call.  A
 * problem whose plan shares tiles over more than 160 CTAs (possible only on a
 * part with more than 160 SMs) is refused with GEMM_ERR_SCRATCH_LIMIT.
 *
 *   - The first call on each device looks up the array's device address (a
 *     runtime query, no allocation) and keeps it for later calls.  Make that
 *     first call before any stream capture on that device.  A device reset
 *     (cudaDeviceReset) makes the kept address stale: do not call this entry
 *     point on that device again in the same process.
 *   - All calls share the one array and it keeps what the last call wrote.
 *     Two calls whose kernels may overlap on the GPU (different streams, or
 *     different host threads, without ordering between them) race on it and
 *     may return wrong results; order them on one stream.
 * Arguments, results and errors otherwise as gemm_f16.
 */
int gemm_f16_noalloc(const gemm_f16_t *A, const gemm_f16_t *B, void *C, int M, int N, int K, int out_dtype,
                     gemm_stream_t stream);

/*
 * Bytes of workspace gemm_f16_ws needs for this problem (0 when its plan
 * uses none), for `num_sms` SMs (0: the current device).
 */
int gemm_f16_workspace_size(int M, int N, int K, int out_dtype, int num_sms, size_t *bytes);

/*
 * The plan gemm_f16 would use for this problem under the current config: the
 * tiling, the grid of output tiles and the sequential K pipeline of "Quickstart:
 * GPU" ("Pipelining: a matmul kernel": grid (m // tile_m, n // tile_n), K /
 * tile_k steps), and the max_concurrent_steps / delay_release pair with the
 * validation and clamping of "JAX Pallas Mosaic GPU 快速上手" ("深入emit_pipeline
 * 的关键参数").  Ragged shapes are planned, not refused: the tile counts are
 * ceilings.  num_sms > 0 plans for that many SMs without touching CUDA
 * (host-only, for tests and tools); num_sms == 0 asks the current device.
 * `out` is caller-owned host memory.
 * Errors: as gemm_f16's argument checks (pointers excepted), GEMM_ERR_NULL
 * for out == NULL, GEMM_ERR_CUDA when num_sms == 0 and no device answers.
 */
int gemm_f16_plan(int M, int N, int K, int out_dtype, int num_sms, gemm_plan *out);

/* The plan gemm_f16_ws would use given a large enough workspace. */
int gemm_f16_plan_ws(int M, int N, int K, int out_dtype, int num_sms, gemm_plan *out);

/* Replace the process-wide tuning config (copied); NULL restores defaults.
 * Its stages and release fields are emit_pipeline's max_concurrent_steps and
 * delay_release ("JAX Pallas Mosaic GPU 快速上手", "深入emit_pipeline的关键参数"),
 * tile_n and tile_k the tile of "Quickstart: GPU" ("Pipelining: a matmul
 * kernel"); as there, stages must exceed release.
 * A call running at the same time on another host thread plans with either
 * the old or the new config, never a mix.
 * Errors: GEMM_ERR_CONFIG for an out-of-range field (the old config stays). */
int gemm_f16_set_config(const gemm_config *cfg);

/* Copy the current tuning config into caller-owned `out`. */
int gemm_f16_get_config(gemm_config *out);

/* Static, NUL-terminated description of a gemm_status code.  No counterpart
 * on the pages (Pallas raises Python exceptions instead). */
const char *gemm_f16_strerror(int code);

/*
 * Synchronise the current device, then report whether any kernel of this
 * library gave up on a bounded wait since the last reset: GEMM_OK or
 * GEMM_ERR_DEVICE_TIMEOUT.  *site (if not NULL) receives which wait gave up
 * first (1 producer/empty slot, 2 MMA/full slot, 3 MMA/free accumulator,
 * 4 epilogue/ready accumulator, 5 drain, 6 split-K partner ready, 7 split-K
 * partials received, 8 stream-K partial flag), 0 if none.  reset != 0 clears it.
 */
int gemm_f16_device_status(int *site, int reset);

/* ABI version of this header: 2 (gemm_plan gained sk_split and sk_helper_tiles). */
int gemm_f16_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_GEMM_F16_H */
