/*
 * gemm_f16_check.h - the bounds-check debug build libtcgemm_check.so (the
 * same sources compiled with -DTCGEMM_CHECK; the product library does not
 * export this entry point).
 *
 * In that build every kernel tests each shared-memory ring, staging and
 * mbarrier address, each Tensor Memory column range and each stream-K
 * workspace slot against its allocation before the access; a failed test
 * skips the access, winds the kernel down through its abort path and leaves a
 * site in the status word gemm_f16_device_status reads: 9 shared memory, 10
 * Tensor Memory, 11 workspace.  It stands in for a memory checker; the pages'
 * counterpart is the silent race the software-pipelining guide warns of when
 * a buffer is reused too early ("JAX Pallas 软件流水线 Software Pipelining 完全
 * 指南", section 9.2, delay_release).
 *
 * The host side of the same tests, on the same arithmetic (csrc/bounds.cuh):
 *
 *   gemm_f16_check_plan(plan, out_dtype, &site)
 *
 * walks every access a launch of `plan` (as gemm_f16_plan or gemm_f16_plan_ws
 * return it; host memory, caller-owned) makes at the level of ring slots,
 * staging buffers, accumulators, split-K blocks and workspace slots, and
 * returns GEMM_OK with *site = 0 when all stay inside their allocations,
 * else GEMM_ERR_CONFIG with *site the first failing site (9, 10 or 11).
 * GEMM_ERR_NULL for a NULL plan or site, GEMM_ERR_DTYPE for a bad out_dtype.
 */
#ifndef TCGEMM_GEMM_F16_CHECK_H
#define TCGEMM_GEMM_F16_CHECK_H

#include "gemm_f16.h"

#ifdef __cplusplus
extern "C" {
#endif

int gemm_f16_check_plan(const gemm_plan *plan, int out_dtype, int *site);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_GEMM_F16_CHECK_H */
