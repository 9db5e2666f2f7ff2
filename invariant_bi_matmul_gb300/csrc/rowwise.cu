// rowwise.cu -- batch-invariant row-wise log-softmax and mean (include/bi_rowwise.h).
//
// Source: book chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Sources (the companion library's mean and log-softmax overrides) and
// Case 6 / The boring rule item 1 (data-parallel rows: one strategy at every batch size).
//
// How a row is cut -- a function of n alone, so the reduction tree is too:
//   * rows up to 262,144 elements live in registers: a cluster of C CTAs (C <= 8) of T
//     threads holds the row, CTA rank r the contiguous segment [r*T*E, (r+1)*T*E), thread
//     t of it the 4-element groups t, t+T, ... (E/4 of them); T, E and C are the smallest
//     that fit (T a power of two in 128..1024, E = 16 or 32).  One read, one write.
//   * longer rows: one CTA of 1024 threads that streams the row once per pass.
// Within a thread, values are folded in ascending group order and ascending element order
// -- a group read as one 128-bit load when the row is aligned, else as scalars, with the
// same arithmetic.  Thread values are combined by a fixed xor butterfly in each warp, then
// over the warp results, then over the cluster's CTAs in ascending rank order (through
// distributed shared memory).  The max is exact in any order.
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "bi.h"
#include "bi_rowwise.h"
#include "common.cuh"
#include "launch.h"

#define BI_EXPORT extern "C" __attribute__((visibility("default")))

namespace bi {

// Defined in api.cu: sets the thread-local message bi_last_error_message() returns.
void set_last_error_message(const char* msg);

namespace {

constexpr int kRowThreads = 1024;
constexpr int kWarps = kRowThreads / 32;

// Elements [4g, 4g+4) of a row, cut at n: exactly the values, in index order, either way.
template <bool BF16>
__device__ __forceinline__ int load_group(const void* row, int g, int n, bool vec, float (&v)[4]) {
    const int i0 = 4 * g;
    const int cnt = n - i0 < 4 ? n - i0 : 4;
    if (BF16) {
        const uint16_t* r = static_cast<const uint16_t*>(row);
        if (vec && cnt == 4) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(r + i0));
            v[0] = __uint_as_float(raw.x << 16);
            v[1] = __uint_as_float(raw.x & 0xffff0000u);
            v[2] = __uint_as_float(raw.y << 16);
            v[3] = __uint_as_float(raw.y & 0xffff0000u);
        } else {
            for (int k = 0; k < cnt; ++k) v[k] = __uint_as_float(uint32_t(r[i0 + k]) << 16);
        }
    } else {
        const float* r = static_cast<const float*>(row);
        if (vec && cnt == 4) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(r + i0));
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
            for (int k = 0; k < cnt; ++k) v[k] = r[i0 + k];
        }
    }
    return cnt;
}

// The CTA-wide combination of one value per thread: xor butterfly in each warp, then over
// the warp results (in warp 0, padded to 32 with the identity), broadcast to every thread.
// MAX: fmaxf (NaN-ignoring, exact); else +.
template <bool MAX>
__device__ __forceinline__ float block_combine(float v, float* scratch) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = MAX ? fmaxf(v, o) : v + o;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // scratch may still be read from the previous combination
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        // lanes past the CTA's warp count contribute the identity (-inf for max, +0 for +)
        v = lane < int(blockDim.x >> 5) ? scratch[lane] : (MAX ? -INFINITY : 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, off);
            v = MAX ? fmaxf(v, o) : v + o;
        }
        if (lane == 0) scratch[kWarps] = v;
    }
    __syncthreads();
    return scratch[kWarps];
}

__global__ void __launch_bounds__(kRowThreads)
log_softmax_kernel(const float* __restrict__ x, int64_t ldx, float* y, int64_t ldy, int n,
                   bool vec_x, bool vec_y) {
    __shared__ float scratch[kWarps + 1];
    pdl_wait();
    pdl_trigger();
    const float* xr = x + int64_t(blockIdx.x) * ldx;
    float* yr = y + int64_t(blockIdx.x) * ldy;
    const int groups = (n + 3) / 4;
    // pass 1: the row max (NaN anywhere makes the whole row NaN, as the definition does)
    float m = -INFINITY;
    bool nan = false;
    for (int g = threadIdx.x; g < groups; g += kRowThreads) {
        float v[4];
        const int cnt = load_group<false>(xr, g, n, vec_x, v);
        for (int k = 0; k < cnt; ++k) {
            nan |= isnan(v[k]);
            m = fmaxf(m, v[k]);
        }
    }
    m = block_combine<true>(m, scratch);
    const bool row_nan = __syncthreads_or(nan);
    // pass 2: sum of exp(x - m)
    float s = 0.f;
    for (int g = threadIdx.x; g < groups; g += kRowThreads) {
        float v[4];
        const int cnt = load_group<false>(xr, g, n, vec_x, v);
        for (int k = 0; k < cnt; ++k) s = s + expf(v[k] - m);
    }
    s = block_combine<false>(s, scratch);
    const float ls = row_nan ? __int_as_float(0x7fc00000) : logf(s);
    // pass 3: y = (x - m) - log(s); every thread reads back exactly the groups it writes,
    // so y may alias x
    for (int g = threadIdx.x; g < groups; g += kRowThreads) {
        float v[4];
        const int cnt = load_group<false>(xr, g, n, vec_x, v);
        for (int k = 0; k < cnt; ++k) v[k] = (v[k] - m) - ls;
        if (vec_y && cnt == 4)
            *reinterpret_cast<float4*>(yr + 4 * g) = make_float4(v[0], v[1], v[2], v[3]);
        else
            for (int k = 0; k < cnt; ++k) yr[4 * g + k] = v[k];
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kRowThreads)
mean_kernel(const void* __restrict__ x, int64_t ldx, int n, bool vec, float* __restrict__ out) {
    __shared__ float scratch[kWarps + 1];
    pdl_wait();
    pdl_trigger();
    const size_t es = BF16 ? 2 : 4;
    const void* xr = static_cast<const char*>(x) + size_t(blockIdx.x) * size_t(ldx) * es;
    const int groups = (n + 3) / 4;
    float s = 0.f;
    for (int g = threadIdx.x; g < groups; g += kRowThreads) {
        float v[4];
        const int cnt = load_group<BF16>(xr, g, n, vec, v);
        for (int k = 0; k < cnt; ++k) s = s + v[k];
    }
    s = block_combine<false>(s, scratch);
    if (threadIdx.x == 0) out[blockIdx.x] = __fdiv_rn(s, float(n));
}

// ------------------------------------------------------ register-resident row kernels

constexpr int kMaxCluster = 8;

struct RowPlan {
    int threads = 0, ept = 0, cluster = 0;  // threads == 0: stream the row instead
};

RowPlan row_plan(int64_t n) {
    RowPlan p;
    for (int ept = 16; ept <= 32; ept *= 2) {
        int t = 128;
        while (t < 1024 && int64_t(t) * ept < n) t *= 2;
        const int64_t c = (n + int64_t(t) * ept - 1) / (int64_t(t) * ept);
        if (c <= kMaxCluster) {
            p.threads = t;
            p.ept = ept;
            p.cluster = int(c);
            return p;
        }
    }
    return p;
}

// Combine one value per CTA across the cluster: every CTA writes its value into slot
// `rank` of every CTA's `slots`, then all fold slots 0..C-1 in order.
template <bool MAX>
__device__ __forceinline__ float cluster_combine(float v, float* slots, int C) {
    if (C == 1) return v;
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0)
        for (int r = 0; r < C; ++r)
            st_cluster_f32(cluster_map(smem_addr(slots + rank), uint32_t(r)), v);
    cluster_sync_all();
    float a = slots[0];
    for (int r = 1; r < C; ++r) a = MAX ? fmaxf(a, slots[r]) : a + slots[r];
    return a;
}

template <int EPT>
__global__ void __launch_bounds__(1024)
log_softmax_reg_kernel(const float* __restrict__ x, int64_t ldx, float* y, int64_t ldy, int n,
                       bool vec_x, bool vec_y, int C) {
    __shared__ float scratch[kWarps + 1];
    __shared__ float x_max[kMaxCluster], x_nan[kMaxCluster], x_sum[kMaxCluster];
    pdl_wait();
    pdl_trigger();
    const int T = int(blockDim.x);
    const int row = int(blockIdx.x) / C;
    const int rank = int(blockIdx.x) - row * C;
    const int seg0 = rank * T * EPT;
    const float* xr = x + int64_t(row) * ldx;
    float* yr = y + int64_t(row) * ldy;
    constexpr int G = EPT / 4;
    // elements of group k held by this thread: e0(k) .. e0(k)+cnt(k)-1
    auto e0 = [&](int k) { return seg0 + 4 * (int(threadIdx.x) + k * T); };
    auto cnt = [&](int k) { return min(max(n - e0(k), 0), 4); };
    float v[EPT];
    float m = -INFINITY;
    bool nan = false;
#pragma unroll
    for (int k = 0; k < G; ++k) {
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        if (cnt(k) > 0) load_group<false>(xr, e0(k) / 4, n, vec_x, w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[4 * k + j] = w[j];
            if (j < cnt(k)) {
                nan |= isnan(w[j]);
                m = fmaxf(m, w[j]);
            }
        }
    }
    m = block_combine<true>(m, scratch);
    m = cluster_combine<true>(m, x_max, C);
    float any_nan = __syncthreads_or(nan) ? 1.f : 0.f;
    any_nan = cluster_combine<true>(any_nan, x_nan, C);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < cnt(k)) s = s + expf(v[4 * k + j] - m);
    s = block_combine<false>(s, scratch);
    s = cluster_combine<false>(s, x_sum, C);
    const float ls = any_nan != 0.f ? __int_as_float(0x7fc00000) : logf(s);
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int c = cnt(k), e = e0(k);
        if (c == 4 && vec_y) {
            *reinterpret_cast<float4*>(yr + e) =
                make_float4((v[4 * k] - m) - ls, (v[4 * k + 1] - m) - ls,
                            (v[4 * k + 2] - m) - ls, (v[4 * k + 3] - m) - ls);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < c) yr[e + j] = (v[4 * k + j] - m) - ls;
        }
    }
}

template <int EPT, bool BF16>
__global__ void __launch_bounds__(1024)
mean_reg_kernel(const void* __restrict__ x, int64_t ldx, int n, bool vec, float* __restrict__ out,
                int C) {
    __shared__ float scratch[kWarps + 1];
    __shared__ float x_sum[kMaxCluster];
    pdl_wait();
    pdl_trigger();
    const int T = int(blockDim.x);
    const int row = int(blockIdx.x) / C;
    const int rank = int(blockIdx.x) - row * C;
    const int seg0 = rank * T * EPT;
    const size_t es = BF16 ? 2 : 4;
    const void* xr = static_cast<const char*>(x) + size_t(row) * size_t(ldx) * es;
    constexpr int G = EPT / 4;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int e0 = seg0 + 4 * (int(threadIdx.x) + k * T);
        if (e0 < n) {
            float w[4];
            const int c = load_group<BF16>(xr, e0 / 4, n, vec, w);
            for (int j = 0; j < c; ++j) s = s + w[j];
        }
    }
    s = block_combine<false>(s, scratch);
    s = cluster_combine<false>(s, x_sum, C);
    if (threadIdx.x == 0 && rank == 0) out[row] = __fdiv_rn(s, float(n));
}

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

constexpr int64_t kI32Max = 0x7fffffffLL;

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace bi

using namespace bi;

BI_EXPORT bi_status bi_log_softmax(const float* x, int64_t ldx, float* y, int64_t ldy,
                                   int64_t rows, int64_t n, bi_stream_t stream) {
    const char* fn = "bi_log_softmax";
    if (rows < 0 || n < 1 || n > kI32Max - 4)
        return fail(BI_ERR_INVALID_ARG, "%s: need rows >= 0 and 1 <= n < 2^31", fn);
    if (ldx < n || ldy < n) return fail(BI_ERR_INVALID_ARG, "%s: ldx and ldy must be >= n", fn);
    if (rows == 0) return BI_OK;
    if (rows > kI32Max) return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    if (!x || !y) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(x, 4) || !aligned(y, 4))
        return fail(BI_ERR_INVALID_ARG, "%s: pointers not element-aligned", fn);
    const bool vec_x = aligned(x, 16) && ldx % 4 == 0;
    const bool vec_y = aligned(y, 16) && ldy % 4 == 0;
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return launched(why, fn);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const RowPlan p = row_plan(n);
    if (p.threads == 0)
        return launched(launch_pdl(log_softmax_kernel, dim3(unsigned(rows)), dim3(kRowThreads),
                                   0, s, x, ldx, y, ldy, int(n), vec_x, vec_y),
                        fn);
    if (rows * p.cluster > kI32Max) return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    const dim3 grid(unsigned(rows * p.cluster)), block(unsigned(p.threads));
    auto k16 = log_softmax_reg_kernel<16>;
    auto k32 = log_softmax_reg_kernel<32>;
    auto kern = p.ept == 16 ? k16 : k32;
    return launched(launch_pdl_cluster(kern, grid, block, 0, s, unsigned(p.cluster), x, ldx, y,
                                       ldy, int(n), vec_x, vec_y, p.cluster),
                    fn);
}

BI_EXPORT bi_status bi_mean(const void* x, int64_t ldx, int x_dtype, int64_t rows, int64_t n,
                            float* out, bi_stream_t stream) {
    const char* fn = "bi_mean";
    if (x_dtype != BI_BF16 && x_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: x_dtype must be BI_BF16 or BI_F32", fn);
    if (rows < 0 || n < 1 || n > kI32Max - 4)
        return fail(BI_ERR_INVALID_ARG, "%s: need rows >= 0 and 1 <= n < 2^31", fn);
    if (ldx < n) return fail(BI_ERR_INVALID_ARG, "%s: ldx < n", fn);
    if (rows == 0) return BI_OK;
    if (rows > kI32Max) return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    if (!x || !out) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    const size_t es = x_dtype == BI_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(out, 4))
        return fail(BI_ERR_INVALID_ARG, "%s: pointers not element-aligned", fn);
    // 4 elements per load: 8 bytes (bf16) or 16 bytes (fp32)
    const bool vec = aligned(x, 4 * es) && (ldx * int64_t(es)) % int64_t(4 * es) == 0;
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return launched(why, fn);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const RowPlan p = row_plan(n);
    if (p.threads == 0) {
        if (x_dtype == BI_BF16)
            return launched(launch_pdl(mean_kernel<true>, dim3(unsigned(rows)),
                                       dim3(kRowThreads), 0, s, x, ldx, int(n), vec, out),
                            fn);
        return launched(launch_pdl(mean_kernel<false>, dim3(unsigned(rows)), dim3(kRowThreads),
                                   0, s, x, ldx, int(n), vec, out),
                        fn);
    }
    if (rows * p.cluster > kI32Max) return fail(BI_ERR_UNSUPPORTED, "%s: too many rows", fn);
    const dim3 grid(unsigned(rows * p.cluster)), block(unsigned(p.threads));
    const unsigned cl = unsigned(p.cluster);
    if (x_dtype == BI_BF16)
        return launched(p.ept == 16
                            ? launch_pdl_cluster(mean_reg_kernel<16, true>, grid, block, 0, s, cl,
                                                 x, ldx, int(n), vec, out, p.cluster)
                            : launch_pdl_cluster(mean_reg_kernel<32, true>, grid, block, 0, s, cl,
                                                 x, ldx, int(n), vec, out, p.cluster),
                        fn);
    return launched(p.ept == 16
                        ? launch_pdl_cluster(mean_reg_kernel<16, false>, grid, block, 0, s, cl, x,
                                             ldx, int(n), vec, out, p.cluster)
                        : launch_pdl_cluster(mean_reg_kernel<32, false>, grid, block, 0, s, cl,
                                             x, ldx, int(n), vec, out, p.cluster),
                    fn);
}
