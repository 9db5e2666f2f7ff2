// glue.cu -- the pointwise decoder glue of the greedy-trace workload (include/bi_glue.h):
// embedding gather, rotary position embedding, SwiGLU gate, residual add and the exact
// greedy argmax.  None of these reduces across rows, so each is batch invariant by
// construction; the argmax reduces within one row under a total order, so its result
// does not depend on the reduction tree either.
//
// All element-wise kernels move 16 bytes (8 bf16) per thread and are HBM bound; they
// follow the same launch discipline as the reductions (programmatic dependent launch,
// device-resident arguments checked in the kernel, never trapping).
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "bi.h"
#include "bi_glue.h"
#include "common.cuh"
#include "launch.h"

#define BI_EXPORT extern "C" __attribute__((visibility("default")))

namespace bi {

// Defined in api.cu: sets the thread-local message bi_last_error_message() returns.
void set_last_error_message(const char* msg);

namespace {

constexpr int kThreads = 256;
constexpr int kArgmaxThreads = 1024;

__device__ __forceinline__ void unpack8(const uint4& raw, float (&v)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 r;
    r.x = pack_bf16x2(v[0], v[1]);
    r.y = pack_bf16x2(v[2], v[3]);
    r.z = pack_bf16x2(v[4], v[5]);
    r.w = pack_bf16x2(v[6], v[7]);
    return r;
}

// ------------------------------------------------------------------------ embedding
__global__ void __launch_bounds__(kThreads)
embedding_kernel(const uint4* __restrict__ table, int vocab, int chunks,
                 const int32_t* __restrict__ ids, int64_t n, uint4* __restrict__ out,
                 int64_t ldo_chunks, unsigned int* err) {
    pdl_wait();
    pdl_trigger();
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= n * chunks) return;
    const int64_t t = idx / chunks;
    const int c = int(idx - t * chunks);
    const int id = ids[t];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (id < 0 || id >= vocab) {
        if (c == 0) latch_error(err, kErrDeviceArg);
    } else {
        v = __ldg(table + int64_t(id) * chunks + c);
    }
    out[t * ldo_chunks + c] = v;
}

// ----------------------------------------------------------------------------- RoPE
// Thread = (token t, head h, group g of 8 pairs): pairs i = 8g .. 8g+7 join elements i
// and i + D/2, i.e. two 16-byte pieces of the head.
__global__ void __launch_bounds__(kThreads)
rope_kernel(uint4* __restrict__ x, int64_t ldx_chunks, int total_q, int heads, int D,
            const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
            float theta, unsigned int* err) {
    pdl_wait();
    pdl_trigger();
    const int groups = D / 16;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= int64_t(total_q) * heads * groups) return;
    const int t = int(idx / (int64_t(heads) * groups));
    const int rem = int(idx - int64_t(t) * heads * groups);
    const int h = rem / groups, g = rem - h * groups;
    int b, qb, j;
    if (cu_q) {
        int lo = 0, hi = B;  // largest b with cu_q[b] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_q[mid] <= t) lo = mid; else hi = mid;
        }
        b = lo;
        j = t - cu_q[b];
        qb = cu_q[b + 1] - cu_q[b];
    } else {
        b = t, j = 0, qb = 1;
    }
    const int L = seq_lens[b];
    if (j < 0 || j >= qb || qb > L) {
        if (h == 0 && g == 0) latch_error(err, kErrDeviceArg);
        return;
    }
    const int pos = L - qb + j;
    uint4* row = x + int64_t(t) * ldx_chunks + (int64_t(h) * D) / 8;
    float lo_v[8], hi_v[8];
    unpack8(row[g], lo_v);
    unpack8(row[D / 16 + g], hi_v);
    float ylo[8], yhi[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int i = 8 * g + e;
        const float inv_freq = powf(theta, -float(2 * i) / float(D));
        float s, c;
        sincosf(float(pos) * inv_freq, &s, &c);
        ylo[e] = lo_v[e] * c - hi_v[e] * s;
        yhi[e] = hi_v[e] * c + lo_v[e] * s;
    }
    row[g] = pack8(ylo);
    row[D / 16 + g] = pack8(yhi);
}

// --------------------------------------------------------------------------- SwiGLU
__global__ void __launch_bounds__(kThreads)
swiglu_kernel(const uint4* gate, int64_t ldg_chunks, const uint4* up, int64_t ldu_chunks,
              uint4* out, int64_t ldo_chunks, int64_t rows, int chunks) {
    // no __restrict__: out may alias gate or up (each thread reads its piece, then writes it)
    pdl_wait();
    pdl_trigger();
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= rows * chunks) return;
    const int64_t r = idx / chunks;
    const int c = int(idx - r * chunks);
    float gv[8], uv[8], y[8];
    unpack8(gate[r * ldg_chunks + c], gv);
    unpack8(up[r * ldu_chunks + c], uv);
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = gv[e] / (1.0f + expf(-gv[e])) * uv[e];
    out[r * ldo_chunks + c] = pack8(y);
}

// ------------------------------------------------------------------------------ add
__global__ void __launch_bounds__(kThreads)
add_kernel(const uint4* a, const uint4* b, uint4* y, int64_t n) {
    // no __restrict__: y may alias a or b (each thread reads its piece, then writes it)
    pdl_wait();
    pdl_trigger();
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t e0 = idx * 8;
    if (e0 >= n) return;
    if (e0 + 8 <= n) {
        float av[8], bv[8], s[8];
        unpack8(a[idx], av);
        unpack8(b[idx], bv);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[e] = av[e] + bv[e];
        y[idx] = pack8(s);
        return;
    }
    const __nv_bfloat16* a16 = reinterpret_cast<const __nv_bfloat16*>(a);
    const __nv_bfloat16* b16 = reinterpret_cast<const __nv_bfloat16*>(b);
    __nv_bfloat16* y16 = reinterpret_cast<__nv_bfloat16*>(y);
    for (int64_t e = e0; e < n; ++e)
        y16[e] = __float2bfloat16_rn(__bfloat162float(a16[e]) + __bfloat162float(b16[e]));
}

// --------------------------------------------------------------------------- argmax
// (value, index) ranked by: any number above NaN; larger value first; lower index first.
// A total order, so every reduction tree picks the same element.
__device__ __forceinline__ bool ranks_above(float va, int ia, float vb, int ib) {
    const bool na = isnan(va), nb = isnan(vb);
    if (na != nb) return nb;
    if (!na && va != vb) return va > vb;
    return ia < ib;
}

__global__ void __launch_bounds__(kArgmaxThreads)
argmax_kernel(const float* __restrict__ logits, int64_t ld, int n, bool vec,
              int32_t* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const float* row = logits + int64_t(blockIdx.x) * ld;
    float best = __int_as_float(0x7fc00000);  // NaN with the largest index: ranks last
    int best_i = 0x7fffffff;
    const int n4 = vec ? (n & ~3) : 0;  // 128-bit loads when every row is 16-byte aligned
    for (int i = threadIdx.x * 4; i < n4; i += kArgmaxThreads * 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(row + i));
        if (ranks_above(v.x, i, best, best_i)) best = v.x, best_i = i;
        if (ranks_above(v.y, i + 1, best, best_i)) best = v.y, best_i = i + 1;
        if (ranks_above(v.z, i + 2, best, best_i)) best = v.z, best_i = i + 2;
        if (ranks_above(v.w, i + 3, best, best_i)) best = v.w, best_i = i + 3;
    }
    for (int i = n4 + int(threadIdx.x); i < n; i += kArgmaxThreads)
        if (ranks_above(row[i], i, best, best_i)) best = row[i], best_i = i;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
        if (ranks_above(ov, oi, best, best_i)) best = ov, best_i = oi;
    }
    __shared__ float s_v[kArgmaxThreads / 32];
    __shared__ int s_i[kArgmaxThreads / 32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) s_v[warp] = best, s_i[warp] = best_i;
    __syncthreads();
    if (warp == 0) {
        best = s_v[lane];
        best_i = s_i[lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, off);
            const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
            if (ranks_above(ov, oi, best, best_i)) best = ov, best_i = oi;
        }
        if (lane == 0) out[blockIdx.x] = best_i;
    }
}

// ------------------------------------------------------------------------ host side
bi_status fail(bi_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_last_error_message(buf);
    return s;
}

bi_status launched(cudaError_t e, const char* fn) {
    if (e == cudaSuccess) return BI_OK;
    return fail(BI_ERR_CUDA, "%s: launch: %s (%s)", fn, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

constexpr int64_t kI32Max = 0x7fffffffLL;

unsigned grid_for(int64_t threads) { return unsigned((threads + kThreads - 1) / kThreads); }

}  // namespace
}  // namespace bi

using namespace bi;

BI_EXPORT bi_status bi_embedding(const void* table, int64_t vocab, int64_t hidden,
                                 const int32_t* ids, int64_t n, void* out, int64_t ldo,
                                 bi_stream_t stream) {
    const char* fn = "bi_embedding";
    if (vocab < 1 || vocab > kI32Max || hidden < 1 || n < 0)
        return fail(BI_ERR_INVALID_ARG, "%s: need vocab in [1, 2^31), hidden >= 1, n >= 0", fn);
    if (ldo < hidden) return fail(BI_ERR_INVALID_ARG, "%s: ldo < hidden", fn);
    if (hidden % 8 || ldo % 8)
        return fail(BI_ERR_UNSUPPORTED, "%s: hidden and ldo must be multiples of 8", fn);
    if (n == 0) return BI_OK;
    if (!table || !ids || !out) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(table) || !aligned16(out) || reinterpret_cast<uintptr_t>(ids) % 4)
        return fail(BI_ERR_UNSUPPORTED, "%s: table and out must be 16-byte aligned", fn);
    if (n * (hidden / 8) > kI32Max * int64_t(kThreads))
        return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return launched(why, fn);
    const int chunks = int(hidden / 8);
    return launched(launch_pdl(embedding_kernel, dim3(grid_for(n * chunks)), dim3(kThreads), 0,
                               reinterpret_cast<cudaStream_t>(stream),
                               static_cast<const uint4*>(table), int(vocab), chunks, ids, n,
                               static_cast<uint4*>(out), ldo / 8, dev->err_word),
                    fn);
}

BI_EXPORT bi_status bi_rope(void* x, int64_t ldx, int64_t total_q, int64_t num_heads,
                            int64_t head_dim, const int32_t* seq_lens, const int32_t* cu_q,
                            int64_t batch, float theta, bi_stream_t stream) {
    const char* fn = "bi_rope";
    if (total_q < 0 || batch < 0 || num_heads < 1)
        return fail(BI_ERR_INVALID_ARG, "%s: negative total_q / batch or num_heads < 1", fn);
    if (head_dim < 16 || head_dim > 256 || head_dim % 16)
        return fail(BI_ERR_UNSUPPORTED, "%s: head_dim must be a multiple of 16 in [16, 256]", fn);
    if (!(theta > 0.0f) || !std::isfinite(theta))
        return fail(BI_ERR_INVALID_ARG, "%s: theta must be finite and > 0", fn);
    if (ldx < num_heads * head_dim) return fail(BI_ERR_INVALID_ARG, "%s: ldx < heads*head_dim", fn);
    if (ldx % 8) return fail(BI_ERR_UNSUPPORTED, "%s: ldx must be a multiple of 8", fn);
    if (total_q == 0) return BI_OK;
    if (batch < 1) return fail(BI_ERR_INVALID_ARG, "%s: tokens without sequences", fn);
    if (!cu_q && total_q != batch)
        return fail(BI_ERR_INVALID_ARG, "%s: without cu_q, total_q must equal batch", fn);
    if (total_q > kI32Max || batch > kI32Max ||
        total_q * num_heads * (head_dim / 16) > kI32Max * int64_t(kThreads))
        return fail(BI_ERR_UNSUPPORTED, "%s: block too large", fn);
    if (!x || !seq_lens) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(x) || reinterpret_cast<uintptr_t>(seq_lens) % 4 ||
        reinterpret_cast<uintptr_t>(cu_q) % 4)
        return fail(BI_ERR_UNSUPPORTED, "%s: x must be 16-byte aligned", fn);
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return launched(why, fn);
    const int64_t threads = total_q * num_heads * (head_dim / 16);
    return launched(launch_pdl(rope_kernel, dim3(grid_for(threads)), dim3(kThreads), 0,
                               reinterpret_cast<cudaStream_t>(stream), static_cast<uint4*>(x),
                               ldx / 8, int(total_q), int(num_heads), int(head_dim), seq_lens,
                               cu_q, int(batch), theta, dev->err_word),
                    fn);
}

BI_EXPORT bi_status bi_swiglu(const void* gate, int64_t ldg, const void* up, int64_t ldu,
                              void* out, int64_t ldo, int64_t rows, int64_t inter,
                              bi_stream_t stream) {
    const char* fn = "bi_swiglu";
    if (rows < 0 || inter < 1) return fail(BI_ERR_INVALID_ARG, "%s: rows < 0 or inter < 1", fn);
    if (ldg < inter || ldu < inter || ldo < inter)
        return fail(BI_ERR_INVALID_ARG, "%s: row strides must be >= inter", fn);
    if (inter % 8 || ldg % 8 || ldu % 8 || ldo % 8)
        return fail(BI_ERR_UNSUPPORTED, "%s: inter and strides must be multiples of 8", fn);
    if (rows == 0) return BI_OK;
    if (!gate || !up || !out) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(gate) || !aligned16(up) || !aligned16(out))
        return fail(BI_ERR_UNSUPPORTED, "%s: pointers must be 16-byte aligned", fn);
    if (rows * (inter / 8) > kI32Max * int64_t(kThreads))
        return fail(BI_ERR_UNSUPPORTED, "%s: too many elements", fn);
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return launched(why, fn);
    const int chunks = int(inter / 8);
    return launched(launch_pdl(swiglu_kernel, dim3(grid_for(rows * chunks)), dim3(kThreads), 0,
                               reinterpret_cast<cudaStream_t>(stream),
                               static_cast<const uint4*>(gate), ldg / 8,
                               static_cast<const uint4*>(up), ldu / 8, static_cast<uint4*>(out),
                               ldo / 8, rows, chunks),
                    fn);
}

BI_EXPORT bi_status bi_add(const void* a, const void* b, void* y, int64_t n, bi_stream_t stream) {
    const char* fn = "bi_add";
    if (n < 0) return fail(BI_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (n == 0) return BI_OK;
    if (!a || !b || !y) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(a) || !aligned16(b) || !aligned16(y))
        return fail(BI_ERR_UNSUPPORTED, "%s: pointers must be 16-byte aligned", fn);
    if ((n + 7) / 8 > kI32Max * int64_t(kThreads))
        return fail(BI_ERR_UNSUPPORTED, "%s: too many elements", fn);
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return launched(why, fn);
    return launched(launch_pdl(add_kernel, dim3(grid_for((n + 7) / 8)), dim3(kThreads), 0,
                               reinterpret_cast<cudaStream_t>(stream), static_cast<const uint4*>(a),
                               static_cast<const uint4*>(b), static_cast<uint4*>(y), n),
                    fn);
}

BI_EXPORT bi_status bi_argmax(const float* logits, int64_t ld, int64_t rows, int64_t n,
                              int32_t* out, bi_stream_t stream) {
    const char* fn = "bi_argmax";
    if (rows < 0 || n < 1 || n > kI32Max - 4 * kArgmaxThreads)
        return fail(BI_ERR_INVALID_ARG, "%s: need rows >= 0 and 1 <= n < 2^31", fn);
    if (ld < n) return fail(BI_ERR_INVALID_ARG, "%s: ld < n", fn);
    if (rows == 0) return BI_OK;
    if (rows > kI32Max) return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    if (!logits || !out) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (reinterpret_cast<uintptr_t>(logits) % 4 || reinterpret_cast<uintptr_t>(out) % 4)
        return fail(BI_ERR_INVALID_ARG, "%s: pointers not element-aligned", fn);
    const bool vec = aligned16(logits) && ld % 4 == 0;
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return launched(why, fn);
    return launched(launch_pdl(argmax_kernel, dim3(unsigned(rows)), dim3(kArgmaxThreads), 0,
                               reinterpret_cast<cudaStream_t>(stream), logits, ld, int(n), vec,
                               out),
                    fn);
}
