/*
 * gemm_f16_trace.h - the event trace of the debug build libtcgemm_trace.so
 * (the same sources compiled with -DTCGEMM_TRACE; the product library does
 * not export this entry point).
 *
 * The pages' counterpart is the profiler switch of Pallas Mosaic GPU's
 * CompilerParams (profile_space, profile_dir: "JAX Pallas Mosaic GPU 快速上手",
 * section "深入emit_pipeline的关键参数"), which records when each warpgroup
 * reaches each point of the pipeline.  Here every kernel launch of the traced
 * library writes, for each of its first `ctas` CTAs and each of six roles
 * (0 producer, 1 MMA issuer, 2..5 epilogue warps), up to `events` records of
 * two 64-bit words:
 *
 *   word 0  the SM clock (clock64), cycles
 *   word 1  bits 63..56: the event code, bits 55..32: its argument,
 *           bits 31..0: for the entry and exit events, %globaltimer modulo
 *           2^32 in nanoseconds (one clock for the whole GPU, read only
 *           there); 0 for every other event
 *
 * A reader places each event in GPU time by its CTA's entry and exit: the
 * SM clock between them maps linearly onto the global timer between them.
 * Event codes (see TraceEvent in csrc/gemm_common.cuh): 1 entry (arg: SM id),
 * 2 set-up done, 3 dependency wait returned, 4 step loads issued (arg: K
 * step), 5 step operands landed (arg: K step), 6 unit's MMAs committed (arg:
 * tile), 7 accumulator ready in the epilogue (arg: tile), 8 split-K partials
 * sent, 9 split-K partials received, 10 stream-K flags seen, 11 chunk store
 * issued (arg: chunk), 12 stores have read their staging, 13 exit, 14 stream-K
 * partial parked.  A role that records more than `events` keeps the first.
 *
 * Launch i (counted from this call) writes slot i % launch_slots of the
 * buffer, laid out [slot][cta][role][event][2 words]: launch_slots * ctas *
 * 6 * events * 16 bytes.  Records never written keep what the caller put
 * there (zero it first: an all-zero record is an empty one).
 */
#ifndef TCGEMM_GEMM_F16_TRACE_H
#define TCGEMM_GEMM_F16_TRACE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Hand the library a device buffer for the trace (NULL stops tracing).
 *   buffer        device memory of at least the size above, 8-byte aligned;
 *                 the caller's, and it must outlive every traced launch
 *   launch_slots  >= 1; ctas >= 1 (CTAs beyond it are not traced); events >= 1
 * Resets the launch count.  Returns GEMM_OK, GEMM_ERR_NULL (bytes too small or
 * a size argument < 1 with a non-NULL buffer) or GEMM_ERR_ALIGN.
 */
int gemm_f16_trace_buffer(void *buffer, size_t bytes, int launch_slots, int ctas, int events);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_GEMM_F16_TRACE_H */
