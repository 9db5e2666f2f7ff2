/*
 * bi_glue.h -- the pointwise decoder glue of the greedy-trace workload, in libbi.
 *
 * The greedy-trace workload runs a Llama-3-8B-shaped decoder stack (hidden 4096, 32
 * query / 8 KV heads, SwiGLU MLP 14336, 8 layers) and asks that its greedy token trace
 * be the same whether tokens are decoded one at a time or verified four at a time, at
 * batch 1, 8 or 32 ([MLX-4279] section Problem: greedy speculative decoding must see
 * identical results for a token alone and inside a verification block; [BOOK] Case 5:
 * the greedy token under three loads).  Besides the reductions of bi.h the stack needs
 * the pointwise operations below.  None of them reduces across rows, so each is batch
 * invariant by construction: output element i depends only on input element(s) i (and,
 * for bi_rope, the token's position; for bi_argmax, its own row).
 *
 * The pages name the stack's shape but define neither the rotary embedding nor the MLP
 * activation; these follow the published definitions: rotary position embedding (Su et
 * al., "RoFormer", 2021) in the rotate-half pairing of the Llama checkpoints, and the
 * SwiGLU gate (Shazeer, "GLU Variants Improve Transformer", 2020).
 *
 * Conventions are those of bi.h: caller-owned device pointers, asynchronous launches on
 * `stream`, argument errors returned before any launch, a device-resident argument out
 * of range (a token id) sets the device error word read by bi_device_status().  Except
 * for bi_argmax, all pointers must be 16-byte aligned and all row strides multiples of
 * 8 elements.
 * Arithmetic is fp32 from bf16 inputs with one round-to-nearest-even to bf16 at the end.
 */
#ifndef BI_GLUE_H_
#define BI_GLUE_H_

#include "bi.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Embedding gather: out[t, :] = table[ids[t], :].
 *   table  bf16 [vocab, hidden] row-major (contiguous rows); hidden % 8 == 0.
 *   ids    int32 [n] (device).  An id outside [0, vocab) writes a zero row and sets
 *          BI_ERR_DEVICE_ARG in the device error word.
 *   out    bf16 [n, hidden], row stride ldo (ldo >= hidden).
 *   Bit-exact copy. */
bi_status bi_embedding(const void* table, int64_t vocab, int64_t hidden, const int32_t* ids,
                       int64_t n, void* out, int64_t ldo, bi_stream_t stream);

/* Rotary position embedding, in place, on a ragged block of tokens.
 *   x        bf16 [total_q, num_heads, head_dim]; token t's heads are contiguous and
 *            start at x + t*ldx (ldx >= num_heads*head_dim).  head_dim % 16 == 0,
 *            head_dim <= 256.
 *   Token positions follow the causal-block rule of bi_verify_block: the tokens of
 *   sequence b are cu_q[b] .. cu_q[b+1]-1 and token j of them sits at position
 *   seq_lens[b] - q_b + j (q_b = cu_q[b+1] - cu_q[b]).  cu_q == NULL means one token
 *   per sequence (token b at position seq_lens[b] - 1), total_q == batch.
 *   Pair i (0 <= i < head_dim/2) joins elements i and i + head_dim/2 and turns by the
 *   angle a = pos * theta^(-2i/head_dim):
 *     y[i] = x[i] cos a - x[i+D/2] sin a,   y[i+D/2] = x[i+D/2] cos a + x[i] sin a.
 *   A token whose sequence index or position is out of range is left unchanged and
 *   sets BI_ERR_DEVICE_ARG. */
bi_status bi_rope(void* x, int64_t ldx, int64_t total_q, int64_t num_heads, int64_t head_dim,
                  const int32_t* seq_lens, const int32_t* cu_q, int64_t batch, float theta,
                  bi_stream_t stream);

/* SwiGLU gate: out[r, i] = silu(gate[r, i]) * up[r, i], silu(g) = g / (1 + exp(-g)).
 *   gate, up  bf16 [rows, inter] with row strides ldg, ldu (>= inter).
 *   out       bf16 [rows, inter] with row stride ldo (>= inter); may alias gate or up
 *             when the strides match. */
bi_status bi_swiglu(const void* gate, int64_t ldg, const void* up, int64_t ldu, void* out,
                    int64_t ldo, int64_t rows, int64_t inter, bi_stream_t stream);

/* Residual add: y[i] = a[i] + b[i] for n contiguous bf16 elements; y may alias a or b. */
bi_status bi_add(const void* a, const void* b, void* y, int64_t n, bi_stream_t stream);

/* Greedy token of each row: out[r] = the index of the largest logits[r, :n], the lowest
 * such index among equal maxima.  NaN ranks below every number (also below -inf), so a
 * NaN is chosen only for an all-NaN row.  This ranking is a total order, so the result
 * is exact and does not depend on the scan order.
 *   logits  fp32 [rows, n], row stride ld (ld >= n); 1 <= n < 2^31.  Rows are read 128
 *           bits at a time when logits is 16-byte aligned and ld % 4 == 0.
 *   out     int32 [rows]. */
bi_status bi_argmax(const float* logits, int64_t ld, int64_t rows, int64_t n, int32_t* out,
                    bi_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_GLUE_H_ */
