/*
 * bi_rowwise.h -- batch-invariant row-wise reductions beyond RMSNorm, in libbi: the
 * log-softmax of a logits row and the mean of a row.
 *
 * Source: book chapter "Batch-invariant kernels: why temperature-0 decoding is still
 * nondeterministic", Sources (the companion library overrides RMSNorm, matmul, mean and
 * log-softmax; log-probabilities are what the chapter's on-policy RL case compares between
 * sampler and trainer, The trap) and Case 6 / The boring rule item 1 (one strategy at
 * every batch size; data-parallel rows).  The pages give no formula beyond the names;
 * these follow the textbook definitions.
 *
 * Construction (both functions): one CTA of 1024 threads per row.  Thread t owns the
 * 4-element groups t, t + 1024, t + 2048, ... of its row and folds them in ascending
 * order (elements within a group in ascending order), whether it reads a group as one
 * 128-bit load (16-byte aligned rows) or as scalars; the 1024 per-thread values are then
 * combined by a fixed butterfly within each warp and a fixed butterfly over the 32 warp
 * results.  The tree therefore depends on n only: a row's bits do not depend on the
 * number of rows, the row's position, its alignment or the stride.
 *
 * Conventions are those of bi.h: caller-owned device pointers, asynchronous launches on
 * `stream`, argument errors returned before any launch.  fp32 arithmetic.
 */
#ifndef BI_ROWWISE_H_
#define BI_ROWWISE_H_

#include "bi.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Log-softmax of each row:
 *   m_r = max_i x[r, i]   (exact),   s_r = sum_i exp(x[r, i] - m_r)   (fp32, tree above),
 *   y[r, i] = (x[r, i] - m_r) - log(s_r).
 *   x  fp32 [rows, n], row stride ldx >= n;  y  fp32 [rows, n], row stride ldy >= n;
 *   y may be x itself (ldy == ldx).  1 <= n < 2^31.  Pointers 4-byte aligned.
 *   A -inf entry gives y = -inf; a row containing NaN, or +inf, or only -inf gives NaN
 *   everywhere in the row (as the definition does). */
bi_status bi_log_softmax(const float* x, int64_t ldx, float* y, int64_t ldy, int64_t rows,
                         int64_t n, bi_stream_t stream);

/* Mean of each row: out[r] = (sum_i x[r, i]) / n, the sum in fp32 by the tree above, the
 * division correctly rounded.
 *   x      [rows, n], dtype x_dtype (BI_BF16 or BI_F32), row stride ldx >= n, aligned to
 *          its element size.  1 <= n < 2^31.
 *   out    fp32 [rows]. */
bi_status bi_mean(const void* x, int64_t ldx, int x_dtype, int64_t rows, int64_t n, float* out,
                  bi_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_ROWWISE_H_ */
