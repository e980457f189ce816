/*
 * ttt_kernels.h — kernel-level entry points of libttt.so, for unit tests and
 * micro-benchmarks of single kernels outside the inner loop.  They compute
 * the same operations the loop uses (see ttt.h for the method); the loop
 * itself never goes through them.
 *
 * All pointers are device memory of the current device; work is issued on
 * `stream` and the call returns without synchronising.  Return value: 0 or a
 * negative TTT_ERR_* code (see ttt.h); a rejected shape is TTT_ERR_SHAPE.
 */
#ifndef TTT_KERNELS_H_
#define TTT_KERNELS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Dense matrix product with fp32 output, the contraction every projection
 * of the decoder block reduces to (a linear layer y = x W^T, its input
 * gradient dx = dy W and its weight gradient dW = dy^T x):
 *   C[m, n] = sum_k A(m, k) B(n, k)  (+ sum_k A(m, k) B2(n, k) if B2)
 *   A(m, k) = a_mn ? A[k*lda + m] : A[m*lda + k]
 *   B(n, k) = b_mn ? B[k*ldb + n] : B[n*ldb + k]   (B2 alike)
 * C is fp32 row-major with row pitch ldc (N and ldc even).
 *   impl 0: tcgen05 tensor cores, A/B/B2 bf16 (lda, ldb multiples of 8,
 *           16-byte aligned bases);
 *   impl 1: SIMT, A/B/B2 bf16;   impl 2: SIMT, A/B/B2 fp32.
 * Accumulation is fp32 in every case. */
int ttt_kernel_gemm(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                    const void* B, int64_t ldb, int32_t b_mn, const void* B2, float* C, int64_t ldc,
                    int32_t impl, void* stream);

/* Error word of the tensor-core kernels launched through this header since
 * the last call (0 = none; otherwise the code of a bounded wait that gave
 * up).  Synchronises the device. */
int ttt_kernel_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TTT_KERNELS_H_ */
