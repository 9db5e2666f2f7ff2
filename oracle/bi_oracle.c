/*
 * bi_oracle.c -- plain, slow, obviously correct CPU oracle for the batch-invariant
 * transformer reductions (matmul, RMSNorm, KV-cache append, decode/verify attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls
 * this file; only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no header, helper, table or constant with the CUDA
 * path.
 *
 * Arithmetic conventions (the pages fix fp32 accumulation and sequential folds):
 *   - bf16 inputs are widened to fp32 exactly (bit shift).
 *   - every reduction is a sequential left fold in fp32, one multiply and one add per
 *     step, never fused: the build uses -ffp-contract=off.  Source: "Batch-invariant
 *     kernels: why temperature-0 decoding is still nondeterministic" (kanthi.in),
 *     Case 2 `sequential` and Case 4 `sum_sq_ordered`.
 *   - bf16 outputs are produced by round-to-nearest-even from the unrounded fp32
 *     result (written out below from the IEEE definition).
 *
 * Parity status: every function here is pinned by a CPU test (printed values from the
 * pages, closed forms, exact-integer cases, fp64 library cross-checks).  None is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------------ */
/* bf16 <-> fp32, from the format definition (1 sign, 8 exponent, 7 mantissa bits). */
/* ------------------------------------------------------------------------------ */

static float bf16_bits_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest, ties-to-even, of an fp32 value to bf16.  NaN stays NaN (quiet). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) {       /* NaN: keep sign, force quiet bit */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) {
        upper += 1u;                             /* carries into exponent correctly */
    }
    return (uint16_t)upper;
}

ORACLE_API void oracle_bf16_round(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_bits(in[i]);
}

ORACLE_API void oracle_bf16_widen(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_to_f32(in[i]);
}

/* ------------------------------------------------------------------------------ */
/* Reduction primitives (book chapter, Cases 1 and 2).                              */
/* ------------------------------------------------------------------------------ */

/* Case 1: left fold in fp64, one binary + at a time, no compensation. */
ORACLE_API double oracle_left_fold_f64(const double* xs, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s = s + xs[i];
    return s;
}

/* Case 2 `sequential`: fp32 left fold starting from +0. */
ORACLE_API float oracle_sum_sequential_f32(const float* a, int64_t n) {
    float s = 0.0f;
    for (int64_t i = 0; i < n; ++i) s = s + a[i];
    return s;
}

/* Case 2 `pairwise`: add adjacent pairs level by level; an odd element at the end
 * of a level is carried unchanged to the next level. */
ORACLE_API float oracle_sum_pairwise_f32(const float* a, int64_t n) {
    if (n <= 0) return 0.0f;
    float* buf = (float*)malloc((size_t)n * sizeof(float));
    if (!buf) return NAN;
    memcpy(buf, a, (size_t)n * sizeof(float));
    int64_t len = n;
    while (len > 1) {
        int64_t out = 0;
        for (int64_t i = 0; i + 1 < len; i += 2) buf[out++] = buf[i] + buf[i + 1];
        if (len % 2) buf[out++] = buf[len - 1];
        len = out;
    }
    float r = buf[0];
    free(buf);
    return r;
}

/* Case 2 `split_k`: contiguous chunks with numpy.array_split sizes (the first
 * n % splits chunks hold one extra element), each folded sequentially, then the
 * partials folded sequentially in chunk order. */
ORACLE_API float oracle_sum_split_f32(const float* a, int64_t n, int64_t splits) {
    if (splits <= 0) return NAN;
    int64_t base = n / splits, extra = n % splits, start = 0;
    float total = 0.0f;
    for (int64_t c = 0; c < splits; ++c) {
        int64_t len = base + (c < extra ? 1 : 0);
        float part = oracle_sum_sequential_f32(a + start, len);
        total = total + part;
        start += len;
    }
    return total;
}

/* Case 4 `sum_sq_ordered` (forward order): s = s + x*x in fp32. */
ORACLE_API float oracle_sum_squares_f32(const float* a, int64_t n) {
    float s = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float sq = a[i] * a[i];
        s = s + sq;
    }
    return s;
}

/* Greedy decoding picks the largest logit; among equal maxima the lowest index. */
ORACLE_API int64_t oracle_argmax_f32(const float* v, int64_t n) {
    /* Greedy decoding picks the largest logit; among equal maxima the lowest index
     * wins.  NaN ranks below every number (below -inf too), so a NaN is picked only
     * when the whole vector is NaN, and then the lowest index.  The pages define no
     * NaN rule; this one makes the choice a total order, independent of scan order. */
    if (n <= 0) return -1;
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i) {
        int best_nan = isnan(v[best]), cur_nan = isnan(v[i]);
        if (best_nan && !cur_nan) best = i;
        else if (!best_nan && !cur_nan && v[i] > v[best]) best = i;
    }
    return best;
}

/* ------------------------------------------------------------------------------ */
/* IEEE binary16 -> fp32, from the format definition (1 sign, 5 exponent bits with  */
/* bias 15, 10 mantissa bits; exponent 0 = subnormal m * 2^-24, 31 = inf/NaN).       */
/* Every binary16 value is exactly representable in fp32.                           */
/* ------------------------------------------------------------------------------ */
static float f16_bits_to_f32(uint16_t h) {
    const unsigned s = (h >> 15) & 1u, e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    float v;
    if (e == 0) v = ldexpf((float)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexpf((float)(m | 0x400u), (int)e - 25);
    return s ? -v : v;
}

ORACLE_API void oracle_f16_widen(const uint16_t* h, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16_bits_to_f32(h[i]);
}

/* widen element i of a 16-bit operand: dtype 0 = bf16 bits, 2 = binary16 bits */
static float widen16(const uint16_t* p, int64_t i, int dtype) {
    return dtype == 2 ? f16_bits_to_f32(p[i]) : bf16_bits_to_f32(p[i]);
}

/* ------------------------------------------------------------------------------ */
/* Matmul: Y[m,n] = sum_k X[m,k] * W(k,n), fp32 accumulation in ascending k.        */
/* W layout 0 ("NK", transposed B, nn.Linear): W(k,n) = w[n*ldw + k].               */
/* W layout 1 ("KN", natural B):              W(k,n) = w[k*ldw + n].                */
/* Output is the unrounded fp32 accumulator (row-major, leading dimension ldy).     */
/* Pages: "Fix/speculative shape invariance" (ml-explore/mlx PR 4279), sections     */
/* Problem and Changes (one reduction order per row, both B orientations); book     */
/* chapter Case 3 (fixed tile, same order at every batch size).                     */
/* ------------------------------------------------------------------------------ */
ORACLE_API void oracle_matmul(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                              int w_layout, float* y, int64_t ldy,
                              int64_t M, int64_t N, int64_t K) {
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float xv = bf16_bits_to_f32(x[m * ldx + k]);
                float wv = bf16_bits_to_f32(w_layout == 0 ? w[n * ldw + k] : w[k * ldw + n]);
                float prod = xv * wv;              /* exact: 8-bit x 8-bit significands */
                acc = acc + prod;
            }
            y[m * ldy + n] = acc;
        }
    }
}

/* The same matmul for 16-bit inputs of either type (dtype 0 = bf16, 2 = binary16).  */
/* A binary16 product is exact in fp32 as well (11-bit x 11-bit significands).      */
ORACLE_API void oracle_matmul16(const uint16_t* x, int64_t ldx, const uint16_t* w, int64_t ldw,
                                int w_layout, float* y, int64_t ldy, int64_t M, int64_t N,
                                int64_t K, int dtype) {
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float xv = widen16(x, m * ldx + k, dtype);
                float wv = widen16(w, w_layout == 0 ? n * ldw + k : k * ldw + n, dtype);
                float prod = xv * wv;
                acc = acc + prod;
            }
            y[m * ldy + n] = acc;
        }
    }
}

/* ------------------------------------------------------------------------------ */
/* RMSNorm (book chapter Case 4, `rms`):                                            */
/*   ss  = sum_i x_i*x_i            (sequential fp32, forward order)                */
/*   inv = 1 / sqrt(ss / H + eps)   (eps inside the root, added to the mean)        */
/*   y_i = (x_i * inv) * gamma_i                                                    */
/* Output: unrounded fp32 rows with leading dimension ldy.                           */
/* ------------------------------------------------------------------------------ */
ORACLE_API void oracle_rmsnorm(const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                               float* y, int64_t ldy, int64_t rows, int64_t H, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * ldx;
        float ss = 0.0f;
        for (int64_t i = 0; i < H; ++i) {
            float v = bf16_bits_to_f32(xr[i]);
            float sq = v * v;
            ss = ss + sq;
        }
        float mean = ss / (float)H;
        float inv = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < H; ++i) {
            float v = bf16_bits_to_f32(xr[i]);
            float t = v * inv;
            y[r * ldy + i] = t * bf16_bits_to_f32(gamma[i]);
        }
    }
}

/* The same RMSNorm for 16-bit x and gamma of either type (0 = bf16, 2 = binary16). */
ORACLE_API void oracle_rmsnorm16(const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                                 float* y, int64_t ldy, int64_t rows, int64_t H, float eps,
                                 int dtype) {
    for (int64_t r = 0; r < rows; ++r) {
        float ss = 0.0f;
        for (int64_t i = 0; i < H; ++i) {
            float v = widen16(x, r * ldx + i, dtype);
            float sq = v * v;
            ss = ss + sq;
        }
        float mean = ss / (float)H;
        float inv = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < H; ++i) {
            float v = widen16(x, r * ldx + i, dtype);
            float t = v * inv;
            y[r * ldy + i] = t * widen16(gamma, i, dtype);
        }
    }
}

/* ------------------------------------------------------------------------------ */
/* Paged KV cache.                                                                  */
/* Cache layout: [num_pages][Hkv][page_size][D] bf16.  Sequence b owns the pages    */
/* block_table[b*max_pages + i], i = 0,1,...; token position p of sequence b lives  */
/* in page block_table[b*max_pages + p/page_size], slot p % page_size.              */
/* A batch of B sequences carries q_b = cu_q[b+1]-cu_q[b] new tokens each (rows     */
/* cu_q[b] .. cu_q[b+1]-1 of the token-major tensors); seq_lens[b] already counts    */
/* them, so new token j of sequence b sits at position seq_lens[b] - q_b + j.       */
/* The book chapter's Case 6 strategy table: the KV cache is updated before the     */
/* attention kernel runs.                                                           */
/* ------------------------------------------------------------------------------ */
static int64_t cache_offset(const int32_t* block_table, int64_t max_pages, int64_t b, int64_t pos,
                            int64_t h, int64_t Hkv, int64_t page_size, int64_t D) {
    int64_t page = block_table[b * max_pages + pos / page_size];
    int64_t slot = pos % page_size;
    return ((page * Hkv + h) * page_size + slot) * D;
}

ORACLE_API void oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new,
                                 uint16_t* k_cache, uint16_t* v_cache,
                                 const int32_t* block_table, int64_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int64_t B,
                                 int64_t Hkv, int64_t D, int64_t page_size) {
    for (int64_t b = 0; b < B; ++b) {
        int64_t q_b = cu_q[b + 1] - cu_q[b];
        for (int64_t j = 0; j < q_b; ++j) {
            int64_t t = cu_q[b] + j;
            int64_t pos = (int64_t)seq_lens[b] - q_b + j;
            for (int64_t h = 0; h < Hkv; ++h) {
                int64_t off = cache_offset(block_table, max_pages, b, pos, h, Hkv, page_size, D);
                memcpy(k_cache + off, k_new + (t * Hkv + h) * D, (size_t)D * sizeof(uint16_t));
                memcpy(v_cache + off, v_new + (t * Hkv + h) * D, (size_t)D * sizeof(uint16_t));
            }
        }
    }
}

/* ------------------------------------------------------------------------------ */
/* Attention for ONE query row (token t of sequence b, query head h):               */
/*   pos  = seq_lens[b] - q_b + j        (causal: the query sees keys 0..pos)       */
/*   s_i  = (sum_d q_d * k_{i,d}) * scale, i = 0..pos   (sequential fp32 over d)     */
/*   m    = max_i s_i                                                               */
/*   p_i  = exp(s_i - m);  l = sum_i p_i  (sequential)                              */
/*   o_d  = (sum_i p_i * v_{i,d}) / l     (sequential over i)                       */
/*   lse  = m + log(l)                                                              */
/* KV head for query head h is h / (Hq/Hkv) (consecutive grouping).                 */
/* This is the plain softmax-attention definition; the split-KV strategy of the     */
/* book chapter's Case 6 reaches the same result up to rounding order.              */
/* ------------------------------------------------------------------------------ */
ORACLE_API int oracle_attention_row(const uint16_t* q, const uint16_t* k_cache,
                                    const uint16_t* v_cache, const int32_t* block_table,
                                    int64_t max_pages, const int32_t* seq_lens,
                                    const int32_t* cu_q, int64_t b, int64_t j,
                                    int64_t Hq, int64_t Hkv, int64_t D, int64_t page_size,
                                    int64_t h, float scale, float* out, float* lse) {
    int64_t q_b = cu_q[b + 1] - cu_q[b];
    int64_t t = cu_q[b] + j;
    int64_t pos = (int64_t)seq_lens[b] - q_b + j;
    int64_t G = Hq / Hkv;
    int64_t hk = h / G;
    int64_t nkeys = pos + 1;
    if (nkeys <= 0) return -1;
    const uint16_t* qv = q + (t * Hq + h) * D;
    float* s = (float*)malloc((size_t)nkeys * sizeof(float));
    float* acc = (float*)malloc((size_t)D * sizeof(float));
    if (!s || !acc) { free(s); free(acc); return -2; }
    float m = -INFINITY;
    for (int64_t i = 0; i < nkeys; ++i) {
        const uint16_t* kv = k_cache + cache_offset(block_table, max_pages, b, i, hk, Hkv, page_size, D);
        float dot = 0.0f;
        for (int64_t d = 0; d < D; ++d) {
            float prod = bf16_bits_to_f32(qv[d]) * bf16_bits_to_f32(kv[d]);
            dot = dot + prod;
        }
        s[i] = dot * scale;
        if (s[i] > m) m = s[i];
    }
    float l = 0.0f;
    for (int64_t d = 0; d < D; ++d) acc[d] = 0.0f;
    for (int64_t i = 0; i < nkeys; ++i) {
        float p = expf(s[i] - m);
        l = l + p;
        const uint16_t* vv = v_cache + cache_offset(block_table, max_pages, b, i, hk, Hkv, page_size, D);
        for (int64_t d = 0; d < D; ++d) {
            float prod = p * bf16_bits_to_f32(vv[d]);
            acc[d] = acc[d] + prod;
        }
    }
    for (int64_t d = 0; d < D; ++d) out[d] = acc[d] / l;
    if (lse) *lse = m + logf(l);
    free(s);
    free(acc);
    return 0;
}

/* All query rows: out [T][Hq][D] fp32 (unrounded), lse [T][Hq] (nullable). */
ORACLE_API int oracle_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                const int32_t* block_table, int64_t max_pages,
                                const int32_t* seq_lens, const int32_t* cu_q, int64_t B,
                                int64_t Hq, int64_t Hkv, int64_t D, int64_t page_size,
                                float scale, float* out, float* lse) {
    for (int64_t b = 0; b < B; ++b) {
        int64_t q_b = cu_q[b + 1] - cu_q[b];
        for (int64_t j = 0; j < q_b; ++j) {
            int64_t t = cu_q[b] + j;
            for (int64_t h = 0; h < Hq; ++h) {
                int rc = oracle_attention_row(q, k_cache, v_cache, block_table, max_pages, seq_lens,
                                              cu_q, b, j, Hq, Hkv, D, page_size, h, scale,
                                              out + (t * Hq + h) * D, lse ? lse + t * Hq + h : NULL);
                if (rc) return rc;
            }
        }
    }
    return 0;
}

/* ============================================================================== */
/* Decoder glue for the greedy-trace workload: a Llama-3-8B-shaped decoder stack   */
/* (hidden 4096, 32 query / 8 KV heads, SwiGLU MLP 14336, 8 layers) whose greedy   */
/* token trace must not depend on batch size or verify width ("Fix/speculative    */
/* shape invariance", section Problem; book chapter Case 5, the greedy token under */
/* three loads).  The pages name the stack's shape but define neither the rotary   */
/* embedding nor the MLP activation; the standard published definitions are used   */
/* (rotary position embedding: Su et al., RoFormer, 2021, in the rotate-half       */
/* pairing of the Llama checkpoints; SwiGLU: Shazeer, "GLU Variants Improve         */
/* Transformer", 2020).  Everything below is evaluated in fp64 and returned        */
/* unrounded; callers narrow to fp32 and then round to bf16 (oracle_bf16_round)   */
/* where the GPU path stores bf16.                                                 */
/* ============================================================================== */

/* Position of token t (0..total-1): tokens of sequence b are cu_q[b]..cu_q[b+1]-1  */
/* and sit at the last q_b positions of its seq_lens[b] tokens.  cu_q == NULL means */
/* one token per sequence (decode).                                                 */
ORACLE_API void oracle_positions(const int32_t* seq_lens, const int32_t* cu_q, int64_t B,
                                 int32_t* pos) {
    for (int64_t b = 0; b < B; ++b) {
        int64_t t0 = cu_q ? cu_q[b] : b;
        int64_t q_b = cu_q ? cu_q[b + 1] - cu_q[b] : 1;
        for (int64_t j = 0; j < q_b; ++j) pos[t0 + j] = (int32_t)(seq_lens[b] - q_b + j);
    }
}

/* Rotary position embedding of x [T][H][D] (row t at x + t*ldx, heads contiguous)  */
/* at positions pos[t].  Pair i (0 <= i < D/2) joins elements i and i + D/2 and is  */
/* turned by the angle pos * theta^(-2i/D):                                          */
/*   y[i]       = x[i] cos(a) - x[i+D/2] sin(a)                                     */
/*   y[i+D/2]   = x[i+D/2] cos(a) + x[i] sin(a)                                     */
ORACLE_API void oracle_rope(const uint16_t* x, int64_t ldx, double* y, int64_t ldy, int64_t T,
                            int64_t H, int64_t D, const int32_t* pos, double theta) {
    int64_t half = D / 2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            const uint16_t* xr = x + t * ldx + h * D;
            double* yr = y + t * ldy + h * D;
            for (int64_t i = 0; i < half; ++i) {
                double freq = pow(theta, -2.0 * (double)i / (double)D);
                double a = (double)pos[t] * freq;
                double c = cos(a), s = sin(a);
                double lo = (double)bf16_bits_to_f32(xr[i]);
                double hi = (double)bf16_bits_to_f32(xr[i + half]);
                yr[i] = lo * c - hi * s;
                yr[i + half] = hi * c + lo * s;
            }
        }
    }
}

/* SwiGLU gating: y = silu(g) * u with silu(g) = g / (1 + exp(-g)). */
ORACLE_API void oracle_swiglu(const uint16_t* g, const uint16_t* u, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        double gv = (double)bf16_bits_to_f32(g[i]);
        double uv = (double)bf16_bits_to_f32(u[i]);
        y[i] = gv / (1.0 + exp(-gv)) * uv;
    }
}

/* Residual add: y = a + b. */
ORACLE_API void oracle_add(const uint16_t* a, const uint16_t* b, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        y[i] = (double)bf16_bits_to_f32(a[i]) + (double)bf16_bits_to_f32(b[i]);
}

/* ------------------------------------------------------------------------------ */
/* Row-wise log-softmax and mean (book chapter "Batch-invariant kernels...",        */
/* Sources: the companion library's mean and log-softmax overrides; the pages name  */
/* the operations only, so these are the textbook definitions, in fp64):            */
/*   log_softmax(x)_i = x_i - m - log(sum_j exp(x_j - m)),  m = max_j x_j          */
/*   mean(x) = (sum_i x_i) / n                                                      */
/* fp32 inputs are widened exactly; bf16 inputs by the bit shift above.             */
/* ------------------------------------------------------------------------------ */
ORACLE_API void oracle_log_softmax_f32(const float* x, int64_t ldx, double* y, int64_t ldy,
                                       int64_t rows, int64_t n) {
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ldx;
        double m = -INFINITY;
        int has_nan = 0;
        for (int64_t i = 0; i < n; ++i) {
            if (isnan(xr[i])) has_nan = 1;
            else if ((double)xr[i] > m) m = (double)xr[i];
        }
        double s = 0.0;
        for (int64_t i = 0; i < n; ++i) s += exp((double)xr[i] - m);
        const double ls = log(s);
        for (int64_t i = 0; i < n; ++i)
            y[r * ldy + i] = has_nan ? NAN : ((double)xr[i] - m) - ls;
    }
}

ORACLE_API void oracle_mean_f32(const float* x, int64_t ldx, int64_t rows, int64_t n,
                                double* out) {
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t i = 0; i < n; ++i) s += (double)x[r * ldx + i];
        out[r] = s / (double)n;
    }
}

ORACLE_API void oracle_mean_bf16(const uint16_t* x, int64_t ldx, int64_t rows, int64_t n,
                                 double* out) {
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t i = 0; i < n; ++i) s += (double)bf16_bits_to_f32(x[r * ldx + i]);
        out[r] = s / (double)n;
    }
}

/* ------------------------------------------------------------------------------ */
/* fp32 inputs ("Fix/speculative shape invariance", ml-explore/mlx PR 4279, the     */
/* tester's comment: f32 dense matmul).  Matmul: the exact sum of the exact          */
/* products of the fp32 inputs, accumulated in fp64 (unrounded reference).           */
/* RMSNorm: the fp32 procedure of oracle_rmsnorm (the book's order) on fp32 inputs. */
/* ------------------------------------------------------------------------------ */
ORACLE_API void oracle_matmul_f32(const float* x, int64_t ldx, const float* w, int64_t ldw,
                                  int w_layout, double* y, int64_t ldy, int64_t M, int64_t N,
                                  int64_t K) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double xv = (double)x[m * ldx + k];
                double wv = (double)(w_layout == 0 ? w[n * ldw + k] : w[k * ldw + n]);
                acc += xv * wv;
            }
            y[m * ldy + n] = acc;
        }
}

ORACLE_API void oracle_rmsnorm_f32(const float* x, int64_t ldx, const float* gamma, float* y,
                                   int64_t ldy, int64_t rows, int64_t H, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        float ss = 0.0f;
        for (int64_t i = 0; i < H; ++i) {
            float v = x[r * ldx + i];
            float sq = v * v;
            ss = ss + sq;
        }
        float mean = ss / (float)H;
        float inv = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < H; ++i) {
            float t = x[r * ldx + i] * inv;
            y[r * ldy + i] = t * gamma[i];
        }
    }
}

/* ------------------------------------------------------------------------------ */
/* Quantized weights ("Fix/speculative shape invariance", ml-explore/mlx PR 4279,   */
/* the tester's comment: affine group sizes 32/64/128, mxfp4, mxfp8, nvfp4; "Fix fp */
/* quantized matmul corruption when the quantized dim is not a multiple of 32",     */
/* Problem: nvfp4 groups of 16 allow K = 16 mod 32).  The pages name the formats;   */
/* the element and scale encodings below follow their published definitions (OCP    */
/* Microscaling formats: FP4 E2M1, FP8 E4M3, E8M0 scales; NVFP4: E2M1 elements with */
/* an FP8 E4M3 scale per 16) and a plain affine code w = scale * q + bias.          */
/* Layout (quantized along K, one row per output column n, "W layout NK"):          */
/*   4-bit codes: byte k/2 of row n, element k in the low nibble when k is even.    */
/*   8-bit codes: byte k of row n.                                                  */
/*   block scales: one byte per block of gs elements, [N][K/gs].                    */
/*   affine: bf16 scale and bias per group of gs, [N][K/gs] each; the dequantized   */
/*   value is fmaf(scale, q, bias) in fp32 rounded to bf16 (nearest even).           */
/* Every other format's dequantized value is exact in bf16.                         */
/* ------------------------------------------------------------------------------ */
enum { Q_MXFP4 = 0, Q_NVFP4 = 1, Q_MXFP8 = 2, Q_AFFINE4 = 3, Q_AFFINE8 = 4 };

static float fp4_e2m1(unsigned c) {  /* sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0 */
    const unsigned e = (c >> 1) & 3u, m = c & 1u;
    const float mag = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, (int)e - 1);
    return (c & 8u) ? -mag : mag;
}

static float fp8_e4m3(unsigned c) {  /* sign bit 7, exponent bits 6-3 (bias 7), mantissa 2-0 */
    const unsigned e = (c >> 3) & 15u, m = c & 7u;
    float mag;
    if (e == 15 && m == 7) mag = NAN;  /* the only NaN pattern; no infinities */
    else if (e == 0) mag = ldexpf((float)m, -9);
    else mag = ldexpf((float)(8u + m), (int)e - 10);
    return (c & 128u) ? -mag : mag;
}

static float scale_e8m0(unsigned c) { return c == 255 ? NAN : ldexpf(1.0f, (int)c - 127); }

ORACLE_API void oracle_decode_fp4(const uint8_t* codes, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp4_e2m1(codes[i] & 15u);
}
ORACLE_API void oracle_decode_fp8(const uint8_t* codes, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = fp8_e4m3(codes[i]);
}
ORACLE_API void oracle_decode_e8m0(const uint8_t* codes, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = scale_e8m0(codes[i]);
}

/* Dequantized W as bf16 bits, [N][K] (row stride K). */
ORACLE_API void oracle_dequantize(const uint8_t* wq, int64_t ldq, const void* scales,
                                  int64_t lds, const uint16_t* biases, int64_t ldb, int format,
                                  int64_t gs, uint16_t* out, int64_t N, int64_t K) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const int64_t g = k / gs;
            unsigned code;
            if (format == Q_MXFP8 || format == Q_AFFINE8) code = wq[n * ldq + k];
            else code = (wq[n * ldq + k / 2] >> ((k & 1) ? 4 : 0)) & 15u;
            float v;
            if (format == Q_MXFP4) v = fp4_e2m1(code) * scale_e8m0(((const uint8_t*)scales)[n * lds + g]);
            else if (format == Q_NVFP4) v = fp4_e2m1(code) * fp8_e4m3(((const uint8_t*)scales)[n * lds + g]);
            else if (format == Q_MXFP8) v = fp8_e4m3(code) * scale_e8m0(((const uint8_t*)scales)[n * lds + g]);
            else {
                const float s = bf16_bits_to_f32(((const uint16_t*)scales)[n * lds + g]);
                const float b = bf16_bits_to_f32(biases[n * ldb + g]);
                v = fmaf(s, (float)code, b);
            }
            out[n * K + k] = f32_to_bf16_bits(v);
        }
}
