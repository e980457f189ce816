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
 *           16-byte aligned bases), tile shape chosen by the planner;
 *   impl 3: as 0 with 128-row tiles on single CTAs;
 *   impl 4: as 0 with 256-row tiles on CTA pairs (cta_group::2);
 *   impl 1: SIMT, A/B/B2 bf16;   impl 2: SIMT, A/B/B2 fp32.
 * Accumulation is fp32 in every case. */
int ttt_kernel_gemm(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                    const void* B, int64_t ldb, int32_t b_mn, const void* B2, float* C, int64_t ldc,
                    int32_t impl, void* stream);

/* Grouped product, the fast MLPs' products when a context holds several
 * sequences (ttt_config.n_seq): `groups` products of group_rows rows each,
 * stacked, each against its own weights:
 *   C[g R + r, n] = sum_k A[g R + r, k] B_g(n, k)  (+ B2_g(n, k) if B2)
 *   R = group_rows, B_g = B + g * group_stride (B2_g alike),
 *   A row-major [groups * R, K] with row pitch lda, B_g(n, k) as B(n, k) of
 *   ttt_kernel_gemm (b_mn, ldb), C fp32 row-major with pitch ldc.
 * impl 0: tensor cores, one launch over every group when the tile height
 * (128, or 256 on CTA pairs) divides R, else one launch per group;
 * impl 3 / 4: as 0 with 128-row tiles / CTA pairs where R allows;
 * impl 1: SIMT.  A, B, B2 bf16 (16-byte aligned, pitches multiples of 8). */
int ttt_kernel_gemm_grouped(int32_t groups, int32_t group_rows, int32_t N, int32_t K, const void* A, int64_t lda,
                            const void* B, int64_t ldb, int32_t b_mn, int64_t group_stride, const void* B2, float* C,
                            int64_t ldc, int32_t impl, void* stream);

/* Weight-gradient product with the fused SGD step of the inner loop (the
 * update of one fast weight, one plain gradient step per chunk):
 *   w32[m, n] -= lr * sum_k A(m, k) B(n, k)
 *   w16[m, n]  = rn_bf16(w32[m, n]);  w16lo[m, n] = rn_bf16(w32 - w16)
 * A(m, k), B(n, k) as in ttt_kernel_gemm (bf16); w32 fp32 and w16 / w16lo
 * bf16, all [M, N] row-major with row pitch ldw (w16 / w16lo may be NULL).
 * impl 0: tcgen05 tensor cores; impl 2: tensor cores on single CTAs;
 * impl 3: tensor cores on CTA pairs (cta_group::2); impl 1: SIMT. */
int ttt_kernel_gemm_sgd(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn, const void* B,
                        int64_t ldb, int32_t b_mn, float* w32, void* w16, void* w16lo, int64_t ldw, float lr,
                        int32_t impl, void* stream);

/* Sliding-window causal attention of one chunk, the attention core of the
 * decoder block (query t sees keys j with t - W < j <= t; grouped KV heads:
 * query head h reads KV head h / (H/Hkv)).  All matrices bf16, device memory:
 *   q     [n, H*hd]        queries of chunk positions pos0 .. pos0+n-1
 *   kring [Hkv, R, hd]     keys by ring slot (position p in slot p mod R)
 *   vring [Hkv, R, hd]     values, same layout
 *   o     [n, H*hd]        output (forward) / forward output (backward)
 *   lse   [H, ld_lse]      fp32 log-sum-exp per (head, row): written by
 *                          the forward, read by the backward
 *   dout  [n, H*hd]        gradient of o (backward)
 *   dqkv  [n, (H+2Hkv)*hd] backward output: dq | dk | dv; dk and dv are the
 *                          gradients of the chunk's own keys and values
 *                          (earlier positions are constants), summed over
 *                          the query heads of each KV head
 *   dsum  [H, ld_lse]      fp32 scratch of the backward (rowsum(dO * O))
 * R must cover W + n - 1 positions.  impl 0: tcgen05 tensor cores
 * (64 <= hd <= 128, hd % 16 == 0, R % 128 == 0, 16-byte aligned bases,
 * else TTT_ERR_SHAPE), kernel variant chosen by size (the forward may split
 * each query tile pair's key range into parts merged by a second kernel,
 * through fp32 scratch allocated per device on first use and kept, so
 * forward calls on one device must not overlap); impl 1: SIMT fp32
 * arithmetic.  Forward only: impl 2 forces the tensor-core kernel with one
 * 128-row query tile per CTA, impl 3 the one with two tiles per CTA and P
 * kept in tensor memory (never split), impl 4 the one-query kernel of a decode step
 * (n == 1, hd a multiple of 32, at most 8 query heads per KV head, q,
 * kring, vring and o 16-byte aligned, else TTT_ERR_SHAPE before any device
 * work; its slice scratch is allocated per device on first use and kept, so
 * calls on one device must not overlap). */
int ttt_kernel_attn_fwd(int32_t impl, int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R,
                        int64_t pos0, const void* q, const void* kring, const void* vring, void* o, float* lse,
                        int32_t ld_lse, void* stream);
int ttt_kernel_attn_bwd(int32_t impl, int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R,
                        int64_t pos0, const void* q, const void* kring, const void* vring, const void* o,
                        const float* lse, int32_t ld_lse, const void* dout, float* dsum, void* dqkv,
                        void* stream);

/* The tensor-core attention backward of ttt_kernel_attn_bwd (impl 0), same
 * arguments and results, but it allocates nothing.  The pages have no
 * counterpart: this entry point exists for callers that must not call
 * cudaMalloc, such as code whose device memory belongs to a caching
 * allocator or a fixed budget (an allocation outside it can fail once that
 * allocator holds the free memory, and escapes its accounting), and
 * real-time callers that plan all memory up front.
 *
 * Its fp32 scratch is a fixed 32 MiB device array inside the library.  Every
 * device context that loads this library's module may reserve it, until the
 * process exits: with lazy module loading (the CUDA default) from the first
 * use of the library on that device, with eager loading when the context is
 * created.  The backward needs 2 * n * H * hd floats of it: larger shapes
 * return TTT_ERR_SHAPE before any device work.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  All
 * calls share the array and it keeps the previous call's contents (nothing
 * in it has to start at zero); calls that overlap on the GPU race on it, so
 * issue them on one stream.  A device-side bounded wait that gives up (not
 * expected) leaves dqkv incomplete and records its code, which the next
 * ttt_kernel_error() returns. */
int ttt_kernel_attn_bwd_noalloc(int32_t n, int32_t H, int32_t Hkv, int32_t hd, int32_t W, int32_t R,
                                int64_t pos0, const void* q, const void* kring, const void* vring, const void* o,
                                const float* lse, int32_t ld_lse, const void* dout, float* dsum, void* dqkv,
                                void* stream);

/* Self-test of the bounded device-side waits every tensor-core kernel uses:
 * launches one CTA whose thread waits on an mbarrier that nothing
 * completes, with a budget of `clocks` SM clocks (1 .. 2e9).  The wait
 * gives up, records its code in the kernel error word and the kernel
 * returns, so the context stays usable.  Returns 0 if the launch went
 * through; read the code with ttt_kernel_error(). */
int ttt_kernel_wait_selftest(int64_t clocks, void* stream);

/* Range checks of the debug build.  libttt_debug.so is this library compiled
 * with TTT_DEBUG_BOUNDS (python -m long_context_lm_ttt_b300.build
 * --debug-bounds).  It range-checks, before each access:
 *   - every tile copy of the tensor-core attention kernels: the inner
 *     coordinate on a 16-byte boundary and inside the tensor, a key/value
 *     box inside one head's ring (query and gradient boxes may start past
 *     the last row, where the copy reads zeros);
 *   - the one-query attention's key/value slice copies, inside the ring and
 *     the pass buffer;
 *   - the decode step's row of the chunk buffers.
 * A failed check records the first violation per source file and skips the
 * access.  A skipped copy makes the kernel abort through its bounded waits;
 * nothing traps.  The context calls (ttt_prefill, ttt_decode, ttt_logits)
 * then return TTT_ERR_INTERNAL naming the kernel.  libttt.so compiles every
 * check away.
 *
 * ttt_kernel_bounds_checked: 1 if this library carries the checks, else 0.
 * ttt_kernel_bounds: synchronises the device, then reads and clears the
 *   records of the current device.  Returns the number of failed checks
 *   since the last call (0: none; always 0 without the checks) or a negative
 *   TTT_ERR_* code.  When the count is positive, *kernel, *index and *limit
 *   (each may be NULL) describe the first failure: the kernel id (1 decode
 *   tail, 2 one-query attention, 3-6 the tensor-core attention forward,
 *   two-tile forward, dq and dk/dv kernels, 7 the self-test), and the index
 *   outside [0, limit).
 * ttt_kernel_bounds_selftest: launches one thread that evaluates one check
 *   on (index, limit) and touches no memory.  With the checks, an index
 *   outside [0, limit) is recorded as kernel 7. */
int ttt_kernel_bounds_checked(void);
int ttt_kernel_bounds(int32_t* kernel, int64_t* index, int64_t* limit);
int ttt_kernel_bounds_selftest(int64_t index, int64_t limit, void* stream);

/* Error word of the tensor-core kernels launched through this header on the
 * current device since the last call, ttt_kernel_attn_bwd_noalloc included
 * (0 = none; otherwise the code of a bounded wait that gave up).  Reading
 * clears it.  Synchronises the device. */
int ttt_kernel_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TTT_KERNELS_H_ */
