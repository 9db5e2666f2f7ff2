/*
 * bi.h -- C ABI of libbi: batch-invariant transformer reductions on one NVIDIA GB300
 * (sm_103a).  Matmul, RMSNorm, paged KV-cache append and decode / speculative-verify
 * attention whose output bits for a given row or query do not depend on how many other
 * rows share the batch, nor on whether a token is evaluated alone or inside a short
 * causal verification block.
 *
 * Sources (web pages this library restates):
 *   [MLX-4279] "Fix/speculative shape invariance", ml-explore/mlx pull request 4279:
 *              sections Problem, Changes and the review thread (limit semantics, both
 *              B orientations, query-length-independent attention split).
 *   [BOOK]     "Batch-invariant kernels: why temperature-0 decoding is still
 *              nondeterministic" (kanthi.in book chapter): Cases 2-5 (reduction trees),
 *              Case 6 strategy table (data-parallel RMSNorm, one matmul config with no
 *              Split-K, fixed split *size* for attention with the cache updated first),
 *              and "The boring rule".
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or retains them.  Host-side state owned by the library: the
 *     batch-invariant limit, a small cache of TMA descriptors (host memory), and one
 *     32-bit device error word per device.
 *   - Every launch is asynchronous and ordered on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream).  Nothing synchronises except bi_device_status().
 *   - bf16 means IEEE bfloat16 stored as 16-bit patterns; outputs are rounded to
 *     nearest-even from an fp32 accumulator.
 *   - Argument errors return BI_ERR_INVALID_ARG (or BI_ERR_UNSUPPORTED for legal but
 *     unimplemented shapes/alignments) BEFORE anything is launched.  A failed launch
 *     returns BI_ERR_CUDA.  Every device-side wait is bounded: a wait that runs out sets
 *     the device error word and the kernel returns; bi_device_status() then reports
 *     BI_ERR_TIMEOUT.  Nothing traps or aborts.  bi_last_error_message() gives a
 *     one-line, thread-local explanation of the last non-OK status.
 *   - Determinism contract: for a fixed library build, every call is deterministic
 *     (same inputs and sizes, same bits).  Calls INSIDE the batch-invariant limit (see
 *     below) are also batch invariant: the bits of output row m of bi_matmul /
 *     bi_rmsnorm depend only on that row's inputs (and W / gamma), never on M, on the
 *     other rows, or on the row's position in the batch; the bits of a query's
 *     attention output depend only on that query, its position and the keys and values
 *     at positions 0..pos of its own sequence -- not on the batch, on the verify-block
 *     width, or on the sequence's total length.  bi_rmsnorm is batch invariant always.
 */
#ifndef BI_H_
#define BI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BI_ABI_VERSION 1

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* bi_stream_t;

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shape      */
    BI_ERR_UNSUPPORTED = 2,  /* legal but not implemented (alignment, head_dim, ...) */
    BI_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed          */
    BI_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out                   */
    BI_ERR_DEVICE_ARG = 5    /* a kernel found a bad device-resident argument
                                (block-table entry out of range, q_len over max_q,
                                seq_len shorter than its block); the work item was
                                skipped, never read or written out of bounds          */
} bi_status;

typedef enum { BI_BF16 = 0, BI_F32 = 1, BI_F16 = 2 } bi_dtype;  /* BI_F16: IEEE binary16 */

typedef enum {
    BI_W_NK = 0,  /* W stored [N, K] row-major ("b_transposed", nn.Linear weight)  */
    BI_W_KN = 1   /* W stored [K, N] row-major (natural orientation)               */
} bi_wlayout;

/* Fixed compile-time constants of this build (they decide the output bits). */
#define BI_PAGE_SIZE 64        /* tokens per KV-cache page                           */
#define BI_ATTN_CHUNK 512      /* keys per split-KV chunk (fixed split size)         */
#define BI_ATTN_MAX_Q 8        /* widest verify block per sequence                   */
#define BI_ATTN_MAX_ROWS 32    /* max q_len * (num_q_heads / num_kv_heads)            */
#define BI_ATTN_MAX_BATCH 1024 /* sequences per attention call                        */

int bi_abi_version(void);
const char* bi_status_string(bi_status s);
/* Thread-local one-line explanation of the last non-OK status returned on this thread. */
const char* bi_last_error_message(void);

/* ---------------------------------------------------------------------------------
 * Batch-invariant limit  [MLX-4279, Changes: set_batch_invariant_limit /
 * get_batch_invariant_limit and the MLX_METAL_BATCH_INVARIANT_LIMIT variable]
 *
 * Process-wide, stored atomically, default 0 (= disabled).  The environment variable
 * BI_BATCH_INVARIANT_LIMIT, if set to a non-negative integer, gives the initial value
 * (read once, at the first call of any entry point).  When the leading dimension
 * (matmul M, RMSNorm rows) or the verify-block width (attention max_q) is <= limit,
 * the entry point MUST use its invariant configuration.  Above the limit, or with the
 * limit at 0, the library picks a faster configuration from the call's sizes, whose
 * bits then depend on those sizes:
 *   - bi_matmul: split-K.  When one 128-row M-tile (M <= 128) leaves SMs idle, a cluster
 *     of up to 8 CTAs shares each output tile, each CTA over a contiguous K range, and
 *     the partials are added in ascending K order (the split count follows N, K, M and
 *     the SM count; see bi_matmul_splits).
 *   - bi_verify_block / bi_decode_attn: the split-KV chunk length (64 .. 2048 keys) is
 *     chosen from the batch, heads, max_seq_len, block width and SM count by a cost
 *     model, among the lengths whose partials fit in the caller's workspace (a
 *     workspace of bi_attn_workspace_size() bytes admits lengths >= BI_ATTN_CHUNK; 8x
 *     that admits all); see bi_attn_chunk.
 *   - bi_rmsnorm has one configuration (already the fastest one).
 * Applications that verify speculative blocks set the limit to cover their largest
 * matmul M (batch x verify width) and their largest verify width.
 * A negative limit returns BI_ERR_INVALID_ARG and leaves the setting unchanged.
 * ------------------------------------------------------------------------------- */
bi_status bi_set_batch_invariant_limit(int64_t limit);
int64_t bi_get_batch_invariant_limit(void);
/* 1 if a call with leading dimension / verify width `dim` falls inside the limit. */
int bi_within_batch_invariant_limit(int64_t dim);

/* ---------------------------------------------------------------------------------
 * Weight prefetch (process-wide, default 0).  Each kernel is launched so that it may
 * start while the previous kernel in its stream is still running; by default it reads
 * no global memory until that kernel has finished.  With the setting at 1, bi_matmul*
 * and bi_qmatmul start streaming W (the codes, scales and biases for bi_qmatmul) before
 * that point, which hides part of the weight stream behind the previous kernel's tail.
 * Set it only if no kernel writes a weight operand right before a call that reads it on
 * the same stream (weights that are fixed for the life of the program qualify; a matmul
 * whose W is the previous matmul's Y does not).  The setting does not change any result.
 * bi_set_weight_prefetch returns BI_ERR_INVALID_ARG for values other than 0 and 1.
 * ------------------------------------------------------------------------------- */
bi_status bi_set_weight_prefetch(int on);
int bi_get_weight_prefetch(void);

/* Introspection (host only, no device access): the configuration a call with these
 * sizes would run under the current limit, on a GPU with num_sms SMs.
 * bi_matmul_splits: CTAs per output tile along K (1 = the invariant single K loop).
 * bi_attn_chunk: split-KV chunk length in keys (BI_ATTN_CHUNK inside the limit);
 *   workspace_bytes is the workspace the call would be given.
 * Both return 0 for invalid sizes. */
int bi_matmul_splits(int64_t M, int64_t N, int64_t K, int w_layout, int num_sms);
int64_t bi_attn_chunk(int64_t batch, int64_t total_q, int64_t max_q, int64_t max_seq_len,
                      int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                      size_t workspace_bytes, int num_sms);

/* ---------------------------------------------------------------------------------
 * bi_matmul  [BOOK Case 3 and Case 6 "Matmul": one compiled config for all shapes, no
 * Split-K; MLX-4279 Problem (GEMV vs gemv_wide vs GEMM by row count is the defect) and
 * review thread (both B orientations)]
 *
 *   Y[m, n] = sum_{k < K} X[m, k] * W(k, n),  fp32 accumulation, then bf16 RNE
 *   (y_dtype BI_BF16) or the fp32 accumulator itself (BI_F32).
 *
 *   x       bf16 [M, K] row-major, row stride ldx elements (ldx >= K).
 *   w       bf16, layout BI_W_NK: [N, K] with row stride ldw (ldw >= K);
 *                 layout BI_W_KN: [K, N] with row stride ldw (ldw >= N).
 *   y       [M, N] row-major, row stride ldy (ldy >= N), dtype y_dtype.
 *   M, N, K >= 0; M = 0 or N = 0 is a no-op; K = 0 writes zeros.
 *   Invariant construction (M inside the batch-invariant limit): one K order for every
 *   M (64-wide K-blocks ascending, four 16-wide kind::f16 steps ascending inside each,
 *   fp32 accumulation in tensor memory, no split of K).  The instruction's height (64
 *   rows for tiles of at most 64 rows, else 128), its width (32 to 256 columns) and the
 *   CTA tile follow M; an element's 16-product step does not depend on them, which the
 *   library's tests check on fp32 output bits at every shape it picks.  Rows beyond M
 *   are never stored.  Outside the limit the K loop may be split
 *   (see the limit section): each part runs the same ascending K order over its range
 *   and the fp32 partials are added in ascending K order before rounding.
 *   Alignment (TMA rule): x, w 16-byte aligned; ldx, ldw multiples of 8 elements;
 *   otherwise BI_ERR_UNSUPPORTED.  y needs only element alignment.
 *   Limits: M, N, K < 2^31.
 * ------------------------------------------------------------------------------- */
bi_status bi_matmul(const void* x, int64_t ldx, const void* w, int64_t ldw, int w_layout,
                    void* y, int64_t ldy, int y_dtype, int64_t M, int64_t N, int64_t K,
                    bi_stream_t stream);

/* bi_matmul with the input type given: in_dtype BI_BF16 or BI_F16 (IEEE binary16) for
 * both x and w (one MMA type for both operands); y_dtype in_dtype (round to nearest even)
 * or BI_F32.  [MLX-4279, the tester's comment: dense matmul divergence also shows for
 * f16 and f32 inputs.]  Same construction, same invariance, same rules as bi_matmul (which
 * is bi_matmul_ex with in_dtype = BI_BF16).
 * in_dtype BI_F32 (y_dtype BI_F32): CUDA cores, each output the fmaf chain over k = 0 ..
 * K-1 in ascending order from +0, for every M and tile; pointers need only element
 * alignment; the batch-invariant limit has no effect (there is one configuration). */
bi_status bi_matmul_ex(const void* x, int64_t ldx, const void* w, int64_t ldw, int w_layout,
                       void* y, int64_t ldy, int in_dtype, int y_dtype, int64_t M, int64_t N,
                       int64_t K, bi_stream_t stream);

/* ---------------------------------------------------------------------------------
 * bi_qmatmul  [MLX-4279, the tester's comment: quantized matmul diverges most with the
 * limit off (affine group sizes 32/64/128, mxfp4, mxfp8, nvfp4); QMM-3912, Problem and
 * Fix: nvfp4's 16-element groups allow K = 16 mod 32, and every tail tile must be
 * bounded (no read of the next row's codes, no store past N)]
 *
 *   Y[m, n] = sum_k X[m, k] * Wd(n, k),  Wd = W dequantized (below) and held as bf16,
 *   fp32 accumulation with the instruction sequence and K order of bi_matmul (layout
 *   NK), then bf16 RNE or fp32.  One configuration: the batch-invariant limit has no
 *   effect, and row m's bits do not depend on M.
 *
 *   x        bf16 [M, K], row stride ldx (16-byte aligned, ldx % 8 == 0).
 *   wq       packed codes, one row per output column n, row stride ldwq bytes (a multiple
 *            of 16; 16-byte aligned):  4-bit formats: byte k/2 holds element k in its low
 *            nibble when k is even, in its high nibble when odd;  8-bit formats: byte k.
 *   scales   one per group of group_size consecutive k of a row, [N][K/group_size], row
 *            stride lds:  BI_Q_MXFP4 / BI_Q_MXFP8: E8M0 bytes (2^(c-127), 255 = NaN);
 *            BI_Q_NVFP4: FP8 E4M3 bytes;  affine: bf16.
 *   biases   affine only: bf16 [N][K/group_size], row stride ldb (else ignored).
 *   Elements: BI_Q_MXFP4, BI_Q_NVFP4: FP4 E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 *   negatives); BI_Q_MXFP8: FP8 E4M3 (0x7F/0xFF NaN, no infinities); affine 4/8-bit:
 *   unsigned integers q.  Dequantized value: element * scale (exact in bf16) for the
 *   block formats; for affine, fmaf(scale, q, bias) in fp32 rounded to bf16.
 *   group_size: 32 (mxfp4, mxfp8), 16 (nvfp4), 32, 64 or 128 (affine); K a multiple of it.
 * ------------------------------------------------------------------------------- */
typedef enum {
    BI_Q_MXFP4 = 0,
    BI_Q_NVFP4 = 1,
    BI_Q_MXFP8 = 2,
    BI_Q_AFFINE4 = 3,
    BI_Q_AFFINE8 = 4
} bi_qformat;
bi_status bi_qmatmul(const void* x, int64_t ldx, const void* wq, int64_t ldwq,
                     const void* scales, int64_t lds, const void* biases, int64_t ldb,
                     int qformat, int group_size, void* y, int64_t ldy, int y_dtype, int64_t M,
                     int64_t N, int64_t K, bi_stream_t stream);

/* bi_qmatmul with the layout of W given  [QMM-3912, Problem and The three defects: the
 * natural-layout kernel (qmm_n) is where the nvfp4 16-column tail was stored out of
 * bounds; MLX-4279 review thread: both B orientations]
 *   w_layout BI_W_NK: as bi_qmatmul.
 *   w_layout BI_W_KN (natural layout, Y = X * Wd with Wd [K, N]): wq holds one row per k,
 *     row stride ldwq bytes, the row's N codes packed as above (4-bit: byte n/2, low
 *     nibble for even n); scales [K][N/group_size] (row stride lds), one per group of
 *     group_size consecutive n of a row; biases likewise.  N must be a multiple of
 *     group_size; K any (rows past K read as zeros).  The dequantized tile is laid out as
 *     bi_matmul's layout-KN W and runs its instruction sequence and K order, so
 *     Y = bi_matmul(x, Wd, BI_W_KN) bit for bit, for every M (one configuration).
 *   Both layouts: every tail tile is bounded (codes past N or K are never read into a
 *   live element, no store past N). */
bi_status bi_qmatmul_ex(const void* x, int64_t ldx, const void* wq, int64_t ldwq,
                        const void* scales, int64_t lds, const void* biases, int64_t ldb,
                        int qformat, int group_size, int w_layout, void* y, int64_t ldy,
                        int y_dtype, int64_t M, int64_t N, int64_t K, bi_stream_t stream);

/* ---------------------------------------------------------------------------------
 * bi_rmsnorm  [BOOK Case 4 (definition and the load-dependent-tree defect) and Case 6
 * "RMSNorm": data-parallel, one row per core, never split]
 *
 *   ss = sum_i x_i^2 (fp32);  y_i = x_i * rsqrt(ss / H + eps) * gamma_i
 *
 *   x      bf16 [rows, H], row stride ldx >= H.   gamma bf16 [H].
 *   y      [rows, H], row stride ldy >= H, dtype y_dtype (bf16 RNE or fp32).
 *   Each row is reduced by exactly one CTA with a reduction tree that is a function of
 *   H only (per-thread ascending sums over 8-element groups, then a fixed warp-shuffle
 *   tree, then a fixed cross-warp tree).  rows = 0 is a no-op.  H in [1, 2^20].
 *   eps must be finite and >= 0.  Any alignment is accepted (16-byte aligned rows use
 *   128-bit loads; the arithmetic is the same either way).
 * ------------------------------------------------------------------------------- */
bi_status bi_rmsnorm(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                     int y_dtype, int64_t rows, int64_t hidden, float eps,
                     bi_stream_t stream);

/* bi_rmsnorm with the input type given: x and gamma both in_dtype (BI_BF16, BI_F16 or
 * BI_F32); y_dtype in_dtype or BI_F32.  Same tree and arithmetic after the exact
 * widening (fp32: the same per-thread groups, butterfly and warp tree on fp32 values). */
bi_status bi_rmsnorm_ex(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                        int in_dtype, int y_dtype, int64_t rows, int64_t hidden, float eps,
                        bi_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Paged KV cache (shared by the three attention entry points)
 *
 *   k_cache, v_cache  bf16 [num_pages, num_kv_heads, BI_PAGE_SIZE, head_dim]; 16-byte
 *                     aligned.
 *   block_table       int32 [batch, max_pages]: block_table[b*max_pages + i] is the
 *                     physical page holding positions [i*PAGE, (i+1)*PAGE) of sequence b.
 *   seq_lens          int32 [batch]: tokens in sequence b INCLUDING its new block.
 *   cu_q              int32 [batch + 1]: new tokens of sequence b are rows
 *                     cu_q[b] .. cu_q[b+1]-1 of the token-major tensors; token j of the
 *                     block sits at position seq_lens[b] - (cu_q[b+1]-cu_q[b]) + j.
 *   All of these are device pointers.  page_size must equal BI_PAGE_SIZE.
 * ------------------------------------------------------------------------------- */

/* bi_kv_append  [BOOK Case 6 "Attention": update the KV cache before the kernel]
 *   Copies k_new / v_new (bf16 [total_q, num_kv_heads, head_dim]) into their slots.
 *   Must run (stream-ordered) before bi_verify_block for the same block. */
bi_status bi_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       int64_t num_pages, const int32_t* block_table, int64_t max_pages,
                       const int32_t* seq_lens, const int32_t* cu_q, int64_t batch,
                       int64_t total_q, int64_t num_kv_heads, int64_t head_dim,
                       int64_t page_size, bi_stream_t stream);

/* Bytes of caller-provided workspace bi_verify_block / bi_decode_attn need: one fp32
 * partial (m, l, o[head_dim]) per (token, query head, chunk), for chunks of
 * BI_ATTN_CHUNK keys up to max_seq_len, rounded up to 16 bytes, then one 4-byte item
 * counter per (token, query head), rounded up to 16 bytes (the counters of one call's
 * (sequence, KV head) pairs: the merge of a pair starts as soon as its chunks are done).
 * The call zeroes the counters itself; no part of the workspace needs initialising.
 * Returns 0 for invalid arguments. */
size_t bi_attn_workspace_size(int64_t total_q, int64_t num_q_heads, int64_t head_dim,
                              int64_t max_seq_len);

/* bi_verify_block  [MLX-4279 Problem/Changes (two-pass SDPA split count must not follow
 * the query length); BOOK Case 6 "Attention" (fixed split size, varying #splits) and
 * the requirement that token 1000 reduces identically with 0 or 999 cached tokens]
 *
 *   For every sequence b and block token j (position pos = seq_lens[b]-q_b+j) and query
 *   head h (KV head h / (num_q_heads/num_kv_heads)):
 *     out[t, h, :] = softmax_i(scale * q[t,h,:] . k_i) @ v_i over keys i = 0..pos
 *     lse[t, h]    = log sum_i exp(scale * q . k_i)            (natural log; nullable)
 *   Split-KV with a FIXED chunk length BI_ATTN_CHUNK counted from key 0 (max_q inside
 *   the batch-invariant limit; outside it the length is chosen per call, see the limit
 *   section): chunk c covers keys [c*CHUNK, (c+1)*CHUNK); a query uses chunks
 *   0..pos/CHUNK, each reduced with the same instruction sequence whatever the batch or
 *   block width, and the partials are merged by log-sum-exp over a fixed tree (eight
 *   contiguous chunk ranges folded in ascending order, then combined in ascending
 *   order) that depends on pos (and the chunk length) alone.
 *
 *   q        bf16 [total_q, num_q_heads, head_dim]; out bf16 same shape; lse fp32
 *            [total_q, num_q_heads] or NULL.  workspace: device memory of at least
 *            bi_attn_workspace_size(total_q, num_q_heads, head_dim, max_seq_len) bytes,
 *            16-byte aligned, contents scratch.  batch <= BI_ATTN_MAX_BATCH.
 *   max_q    upper bound of every q_b (1..BI_ATTN_MAX_Q), max_q * (num_q_heads /
 *            num_kv_heads) <= BI_ATTN_MAX_ROWS.  max_seq_len: upper bound of every
 *            seq_lens[b] (>= 1).  head_dim in {64, 128}.  num_q_heads % num_kv_heads == 0.
 *   Device-resident arguments are checked in the kernel (page index < num_pages,
 *   1 <= q_b <= max_q, q_b <= seq_len <= max_seq_len); an offending work item is skipped
 *   and BI_ERR_DEVICE_ARG is latched for bi_device_status(). */
bi_status bi_verify_block(const void* q, const void* k_cache, const void* v_cache,
                          int64_t num_pages, const int32_t* block_table, int64_t max_pages,
                          const int32_t* seq_lens, const int32_t* cu_q, int64_t batch,
                          int64_t total_q, int64_t max_q, int64_t max_seq_len,
                          int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                          int64_t page_size, float scale, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* bi_decode_attn: bi_verify_block with exactly one new token per sequence (token b is
 * the last position of sequence b; q, out: [batch, num_q_heads, head_dim]).  Runs the
 * same kernels, so its bits equal bi_verify_block's with q_b = 1. */
bi_status bi_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                         int64_t num_pages, const int32_t* block_table, int64_t max_pages,
                         const int32_t* seq_lens, int64_t batch, int64_t max_seq_len,
                         int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                         int64_t page_size, float scale, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* bi_prefill_attn  [BOOK Case 6 "Attention" and the paragraph after its table: serving
 * engines slice sequences (chunked prefill, prefix caching), and token 1000 must reduce
 * identically whether 0 or 999 tokens are already cached -- one loop over cache and new
 * tokens]
 *
 *   bi_verify_block for blocks of any width: a prompt cut into chunks of any sizes, each
 *   chunk's K/V appended (bi_kv_append) before its call, or a prompt continuing a cached
 *   prefix.  Every query is reduced exactly as bi_verify_block / bi_decode_attn reduce
 *   it inside the batch-invariant limit (chunk length BI_ATTN_CHUNK, the same
 *   per-page steps, the same merge tree), so its out and lse bits do not depend on how
 *   the sequence was split into calls or on the other queries of the call.  The limit
 *   has no effect (one configuration).
 *
 *   Arguments as bi_verify_block, except: max_q >= 1 without upper bound, and
 *   num_q_heads / num_kv_heads must divide 128 (a tile is 128 query rows: 128 / G tokens
 *   times the G query heads of one KV head).  Workspace: bi_attn_workspace_size(total_q,
 *   num_q_heads, head_dim, max_seq_len) bytes.  Device-resident arguments are checked as
 *   in bi_verify_block. */
bi_status bi_prefill_attn(const void* q, const void* k_cache, const void* v_cache,
                          int64_t num_pages, const int32_t* block_table, int64_t max_pages,
                          const int32_t* seq_lens, const int32_t* cu_q, int64_t batch,
                          int64_t total_q, int64_t max_q, int64_t max_seq_len,
                          int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                          int64_t page_size, float scale, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* ---------------------------------------------------------------------------------
 * bi_verify_block_static_ws -- bi_verify_block without a caller-provided workspace.
 * (No counterpart on the pages; it exists for callers that cannot allocate.)
 *
 * For callers that cannot call cudaMalloc where they run attention (code recorded into
 * or replayed from someone else's CUDA graph, allocator-free runtimes that only hand
 * over the tensors they own, real-time paths where an allocation and its implicit
 * synchronisation are not allowed).  Same arguments as bi_verify_block minus
 * workspace / workspace_bytes, and the same results as bi_verify_block given a workspace
 * of exactly bi_attn_workspace_size(total_q, num_q_heads, head_dim, max_seq_len) bytes
 * (outside the batch-invariant limit the chunk length depends on the workspace size, so
 * that size is what this entry point passes on).  The workspace is a fixed device array
 * of BI_STATIC_WS_BYTES inside the library, present on every GPU that loads it until the
 * process exits.  Nothing is allocated.
 *   - A block whose bi_attn_workspace_size(...) exceeds BI_STATIC_WS_BYTES is refused
 *     with BI_ERR_UNSUPPORTED (message names both sizes); use bi_verify_block then.  This
 *     size check comes first, so a call whose sizes are both invalid and too large is
 *     reported as BI_ERR_UNSUPPORTED; the other arguments are checked as in
 *     bi_verify_block.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) and keeps it for the life of the process; make that first
 *     call before any stream capture.  After cudaDeviceReset (or anything else that
 *     destroys the device's primary context) the kept address is stale: a process that
 *     resets a device must not call this entry point again.
 *   - Every call shares the one array and it keeps the last call's contents (nothing in
 *     it needs to start at zero).  Calls whose kernels overlap on the GPU -- different
 *     streams, different host threads -- race on it: serialise them.
 * ------------------------------------------------------------------------------- */
#define BI_STATIC_WS_BYTES (32u * 1024u * 1024u)
bi_status bi_verify_block_static_ws(const void* q, const void* k_cache, const void* v_cache,
                                    int64_t num_pages, const int32_t* block_table,
                                    int64_t max_pages, const int32_t* seq_lens,
                                    const int32_t* cu_q, int64_t batch, int64_t total_q,
                                    int64_t max_q, int64_t max_seq_len, int64_t num_q_heads,
                                    int64_t num_kv_heads, int64_t head_dim, int64_t page_size,
                                    float scale, void* out, float* lse, bi_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Device error word
 * bi_device_status synchronises `stream`, reads and clears the current device's error
 * word and returns BI_OK, BI_ERR_TIMEOUT (a bounded wait ran out), BI_ERR_DEVICE_ARG,
 * or BI_ERR_CUDA if the synchronisation itself failed.
 * ------------------------------------------------------------------------------- */
bi_status bi_device_status(bi_stream_t stream);

/* Failure-detection self-test: launches one CTA that waits on an mbarrier nobody
 * arrives at, bounded by timeout_ns nanoseconds (1e3 .. 1e10).  The wait runs out, the
 * kernel latches BI_ERR_TIMEOUT in the error word and returns, leaving the context
 * usable.  Used by the tests to exercise the timeout path without faulting a GPU. */
bi_status bi_selftest_wait_timeout(uint64_t timeout_ns, bi_stream_t stream);

/* Failure-detection self-test of the real kernels: sets the budget of every bounded wait
 * in the GEMM, attention and prefill kernels (and the merge) of the current device to
 * timeout_ns nanoseconds (1e3 .. 1e10), or back to the library default (about 4 s) with
 * 0.  Stream-ordered (kernels issued on `stream` after the call see it; the call
 * synchronises `stream`).  With a budget shorter than a call's runtime the call's waits
 * run out: the kernels latch BI_ERR_TIMEOUT in the error word, raise their CTA's abort
 * flag, let the copies and MMAs already issued complete (each such drain bounded by
 * 100 ms, not by this budget), free tensor memory and return, leaving the context
 * usable.  The outputs of a call that timed out are undefined.  Process-wide per device;
 * for tests only.  BI_ERR_INVALID_ARG for other values. */
bi_status bi_selftest_set_wait_budget(uint64_t timeout_ns, bi_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BI_H_ */
