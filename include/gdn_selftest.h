/*
 * gdn_selftest.h — diagnostic entry point of libgdn.so (not part of the GDN
 * path): checks the tensor-core building block that the chunked prefill uses.
 * The pages define no such operation; it exists so the tcgen05 operand
 * layout can be tested against a plain host GEMM.
 */
#ifndef GDN_SELFTEST_H
#define GDN_SELFTEST_H

#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * D[128][N] = A[128][K] * B[N][K]^T with bf16 A, B (row-major, device) and f32
 * D (row-major, device), computed by one thread block with tcgen05.mma from
 * shared memory into TMEM. N in {16, 32, ..., 256}, K in {16, 32, ..., 128}.
 * dev_err (device, nullable) receives bit 1 if the completion wait timed out.
 * starve_wait = 1 exercises that failure path without any fault: the MMAs'
 * completion is not attached to the barrier the block waits on, so the
 * bounded wait gives up, sets bit 1, then attaches and drains the MMAs,
 * frees its TMEM and returns (D is left unwritten).
 * Returns GDN_ERR_INVALID for other shapes, GDN_ERR_CUDA on launch failure.
 */
gdn_status gdn_selftest_tc_gemm(const uint16_t* A, const uint16_t* B, float* D, int32_t N,
                                int32_t K, int32_t starve_wait, uint32_t* dev_err, void* stream);

/*
 * D[128][N] = A[128][K] * B[N][K]^T with f32 A, B and D (row-major, device) on
 * the tf32 tensor-core path (tcgen05.mma kind::tf32), one thread block.
 * N in {16, 32, ..., 256}, K in {8, 16, ..., 128}. dev_err (device, nullable)
 * receives bit 1 if the completion wait timed out. Same error returns as above.
 */
gdn_status gdn_selftest_tc_gemm_tf32(const float* A, const float* B, float* D, int32_t N,
                                     int32_t K, uint32_t* dev_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SELFTEST_H */
