/* C ABI of the sm_103a row softmax (libgemm_sm103.so).
 *
 * The operation is the fused row softmax of "02: Fused softmax"
 * (phobos-lang.dev tutorial, the `softmax` kernel and the prose above it):
 * for every row i of an fp32 array, over the first n columns,
 *     m_i = max_j X[i,j],   Y[i,j] = exp(X[i,j] - m_i) / sum_k exp(X[i,k] - m_i).
 * The tutorial stores rows wider than n (its 781-column rows are 784 wide)
 * and leaves the columns past n out of the maximum and the sum; here they
 * are neither read nor written.
 *
 * Status codes are those of gemm_sm103.h (gemm_status_t); the last CUDA
 * error of a failed launch is reported by gemm_last_cuda_error().
 */
#ifndef SOFTMAX_SM103_H
#define SOFTMAX_SM103_H

#include <stdint.h>

#include "gemm_sm103.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Longest row (columns) the kernels hold: one thread-block cluster of eight
 * CTAs keeps 65,536 fp32 values in registers. */
#define SOFTMAX_MAX_COLS 65536

/* Y = softmax of each row of X, along the row.
 *
 *   X    device pointer, fp32, row-major: row i starts at X + i*ldx. Read only.
 *   ldx  row pitch of X in elements, ldx >= n.
 *   Y    device pointer, fp32, row-major with pitch ldy >= n. Only Y[i, 0..n)
 *        is written; the columns past n keep their contents.
 *   M    rows (M >= 0); n columns of each row (0 <= n <= SOFTMAX_MAX_COLS).
 *   stream  cudaStream_t (NULL = the legacy default stream); the work is
 *        enqueued there without host synchronisation.
 *
 * Ownership: the caller owns X and Y; the library allocates nothing.
 * In place: Y == X with ldy == ldx is allowed (a row is read whole before
 * any of it is written). Any other overlap of the byte ranges the two
 * arrays span gives GEMM_ERR_INVALID_ARG.
 * Errors (synchronous, nothing enqueued): M < 0, n < 0, ldx < n, ldy < n,
 * a NULL pointer with M > 0 and n > 0, or an overlap -> GEMM_ERR_INVALID_ARG;
 * n > SOFTMAX_MAX_COLS, a pitch above 2^31, or X / Y not 4-byte aligned ->
 * GEMM_ERR_UNSUPPORTED; a failed launch -> GEMM_ERR_CUDA. M == 0 or n == 0
 * is a no-op returning GEMM_OK.
 * Rows start on 16-byte boundaries when X and Y are 16-byte aligned and
 * both pitches are multiples of 4; the kernels then move float4 vectors,
 * otherwise single floats. */
int softmax_rows_f32(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M, int64_t n, void* stream);

/* The launch softmax_rows_f32 makes for M rows of n columns on the current
 * device: threads per row (32 = one warp per row), CTAs per row (the
 * cluster size, 1 = no cluster) and CTAs in the grid. Any output may be NULL.
 * Errors: M < 0, n < 1 -> GEMM_ERR_INVALID_ARG; n > SOFTMAX_MAX_COLS ->
 * GEMM_ERR_UNSUPPORTED; a failed device query -> GEMM_ERR_CUDA. */
int softmax_rows_plan(int64_t M, int64_t n, int32_t* threads_per_row, int32_t* cluster_ctas, int32_t* grid_ctas);

/* Number of softmax kernel launches this process has made (all devices). */
uint64_t softmax_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SOFTMAX_SM103_H */
