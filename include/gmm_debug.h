/*
 * gmm_debug.h - test-only entry points of libgmm.  Not part of the EM API.
 */
#ifndef GMM_DEBUG_H
#define GMM_DEBUG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gmm_debug_tc_gemm - checks the tensor-core building blocks the fused
 * kernels use (128-byte swizzled K-major shared-memory operands, tcgen05.mma
 * kind::f16 into tensor memory, completion through an mbarrier, tcgen05.ld).
 * C[128][n] = A[128][kdim] * B[n][kdim]^T with A, B row-major fp16 bits
 * (device), C row-major fp32 (device).  kdim in {64, 128, 256}, or one of
 * those + 16: the last 16 columns are then staged in the unswizzled K = 16
 * layout (8-row x 16-byte core matrices) and contracted by one more MMA.  n
 * in {64, 128}.  One thread block; asynchronous on `stream`.  *status_dev (device
 * int32, zeroed by the caller) becomes 6 (GMM_ERR_TIMEOUT) if the bounded
 * wait for the MMA ran out.  Returns 0, 1 for bad arguments, 7 for a CUDA
 * error.
 */
int gmm_debug_tc_gemm(const void* A, const void* B, float* C, int kdim, int n,
                      int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GMM_DEBUG_H */
