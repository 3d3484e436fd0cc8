/*
 * add_matrices.h - C ABI of the pipelined blocked add, the second workload on
 * the GEMM library's pipeline machinery.
 *
 * The operation is add_matrices of "JAX Pallas 软件流水线 Software Pipelining
 * 完全指南", section 6: Z = X + Y for f32 arrays, computed block by block with
 * the copies of the next blocks overlapping the current addition, and
 * checked there with assert_array_equal against x + y.  Each element is one
 * IEEE binary32 addition (round to nearest even), so the result is bit-exact
 * whatever the blocking.
 *
 * Status codes are gemm_status's (gemm_f16.h); gemm_f16_strerror describes
 * them and gemm_f16_device_status reports a device-side timeout.
 */
#ifndef TCGEMM_ADD_MATRICES_H
#define TCGEMM_ADD_MATRICES_H

#include "gemm_f16.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Z = X + Y, element by element.
 *
 *   X, Y   device, M x N f32, row-major (row stride N), 16-byte aligned, read-only
 *   Z      device, M x N f32, row-major, 16-byte aligned; may be X or Y itself
 *          (in place) but may not partly overlap either
 *   M, N   >= 0, N a multiple of 4 (16-byte rows for TMA); M == 0 or N == 0
 *          is a no-op
 *   stream the call is asynchronous on it
 * Errors: GEMM_ERR_DIM, GEMM_ERR_NULL, GEMM_ERR_ALIGN, GEMM_ERR_ALIAS before any
 * CUDA call; GEMM_ERR_CUDA, GEMM_ERR_ARCH, GEMM_ERR_TMAP, GEMM_ERR_LAUNCH after.
 */
int add_matrices_f32(const float *X, const float *Y, float *Z, int M, int N, gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_ADD_MATRICES_H */
