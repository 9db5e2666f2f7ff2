// api.cu -- the C ABI of libbi (declared in include/bi.h): argument validation, the
// process-wide batch-invariant limit, the per-device error word and the dispatch to the
// kernel launchers.  No entry point allocates device memory.
#include <atomic>
#include <cerrno>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "bi.h"
#include "launch.h"

#define BI_EXPORT extern "C" __attribute__((visibility("default")))

namespace bi {

// One 32-bit error word per device (bits: kErrTimeout, kErrDeviceArg).  Host code only
// ever uses the address obtained from cudaGetSymbolAddress for the current device.
// Per device: the error word (element 0) and, as the 64-bit word at elements 2..3, the
// budget of the kernels' bounded waits in ns (0 = the default; only a self-test sets it).
__device__ __align__(16) unsigned int g_error_block[4];

namespace {

thread_local std::string t_last_message;

bi_status fail(bi_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_message = buf;
    return s;
}

bi_status cuda_fail(cudaError_t e, const char* what) {
    if (e == cudaErrorNotSupported)
        return fail(BI_ERR_UNSUPPORTED, "%s: shape or pointer layout not supported", what);
    return fail(BI_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ------------------------------------------------------------------ limit (atomic)
std::atomic<int64_t> g_limit{0};
// early weight reads (bi_set_weight_prefetch); off: every kernel waits for the previous
// grid in its stream before it reads global memory
std::atomic<int> g_weight_prefetch{0};
std::once_flag g_limit_once;

void init_limit_from_env() {
    std::call_once(g_limit_once, []() {
        const char* v = std::getenv("BI_BATCH_INVARIANT_LIMIT");
        if (!v || !*v) return;
        char* end = nullptr;
        errno = 0;
        long long x = std::strtoll(v, &end, 10);
        if (errno == 0 && end && *end == '\0' && x >= 0) g_limit.store(x);
    });
}

// ------------------------------------------------------------ device bookkeeping
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_devs[kMaxDevices];

constexpr int64_t kI32Max = 0x7fffffffLL;

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

void set_last_error_message(const char* msg) { t_last_message = msg ? msg : ""; }

const DeviceInfo* current_device_info(cudaError_t* why) {
    int d = -1;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
        if (why) *why = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& di = g_devs[d];
    if (di.device < 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
        void* word = nullptr;
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&word, g_error_block);
        if (e == cudaSuccess) e = cudaMemset(word, 0, sizeof(g_error_block));
        if (e != cudaSuccess) {
            if (why) *why = e;
            return nullptr;
        }
        di.num_sms = sms;
        di.err_word = static_cast<unsigned int*>(word);
        di.device = d;
    }
    return &di;
}

}  // namespace bi

using namespace bi;

// ==================================================================== misc / limit

BI_EXPORT int bi_abi_version(void) { return BI_ABI_VERSION; }

BI_EXPORT const char* bi_status_string(bi_status s) {
    switch (s) {
        case BI_OK: return "BI_OK";
        case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
        case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED";
        case BI_ERR_CUDA: return "BI_ERR_CUDA";
        case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT";
        case BI_ERR_DEVICE_ARG: return "BI_ERR_DEVICE_ARG";
    }
    return "BI_ERR_UNKNOWN";
}

BI_EXPORT const char* bi_last_error_message(void) { return t_last_message.c_str(); }

BI_EXPORT bi_status bi_set_batch_invariant_limit(int64_t limit) {
    init_limit_from_env();
    if (limit < 0) return fail(BI_ERR_INVALID_ARG, "batch-invariant limit must be >= 0");
    g_limit.store(limit);
    return BI_OK;
}

BI_EXPORT int64_t bi_get_batch_invariant_limit(void) {
    init_limit_from_env();
    return g_limit.load();
}

BI_EXPORT bi_status bi_set_weight_prefetch(int on) {
    if (on != 0 && on != 1) return fail(BI_ERR_INVALID_ARG, "weight prefetch must be 0 or 1");
    g_weight_prefetch.store(on);
    return BI_OK;
}

BI_EXPORT int bi_get_weight_prefetch(void) { return g_weight_prefetch.load(); }

BI_EXPORT int bi_within_batch_invariant_limit(int64_t dim) {
    init_limit_from_env();
    const int64_t lim = g_limit.load();
    return lim > 0 && dim <= lim ? 1 : 0;
}

BI_EXPORT int bi_matmul_splits(int64_t M, int64_t N, int64_t K, int w_layout, int num_sms) {
    if (M < 1 || N < 1 || K < 1 || M > kI32Max || N > kI32Max || K > kI32Max || num_sms < 1 ||
        (w_layout != BI_W_NK && w_layout != BI_W_KN))
        return 0;
    const bool split_ok = !bi_within_batch_invariant_limit(M);
    return gemm_schedule(M, N, K, w_layout == BI_W_KN, num_sms, split_ok).splits;
}

BI_EXPORT int64_t bi_attn_chunk(int64_t batch, int64_t total_q, int64_t max_q,
                                int64_t max_seq_len, int64_t num_q_heads, int64_t num_kv_heads,
                                int64_t head_dim, size_t workspace_bytes, int num_sms) {
    if (batch < 1 || total_q < batch || max_q < 1 || total_q > batch * max_q ||
        max_seq_len < 1 || num_kv_heads < 1 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || (head_dim != 64 && head_dim != 128) || num_sms < 1)
        return 0;
    PagedArgs a{};
    a.batch = batch;
    a.total_q = total_q;
    a.max_q = max_q;
    a.max_seq_len = max_seq_len;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.head_dim = head_dim;
    return int64_t(1) << attn_chunk_log2(a, workspace_bytes, num_sms,
                                         bi_within_batch_invariant_limit(max_q) != 0);
}

// ========================================================================== matmul

namespace {

bi_status matmul_impl(const char* fn, const void* x, int64_t ldx, const void* w, int64_t ldw,
                      int w_layout, void* y, int64_t ldy, int in_dtype, int y_dtype, int64_t M,
                      int64_t N, int64_t K, bi_stream_t stream) {
    init_limit_from_env();
    if (M < 0 || N < 0 || K < 0) return fail(BI_ERR_INVALID_ARG, "%s: negative M/N/K", fn);
    if (M > kI32Max || N > kI32Max || K > kI32Max)
        return fail(BI_ERR_UNSUPPORTED, "%s: M, N, K must be < 2^31", fn);
    if (w_layout != BI_W_NK && w_layout != BI_W_KN)
        return fail(BI_ERR_INVALID_ARG, "%s: w_layout must be BI_W_NK or BI_W_KN", fn);
    if (in_dtype != BI_BF16 && in_dtype != BI_F16 && in_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: in_dtype must be BI_BF16, BI_F16 or BI_F32", fn);
    if (y_dtype != in_dtype && y_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: y_dtype must be in_dtype or BI_F32", fn);
    if (M == 0 || N == 0) return BI_OK;
    if (in_dtype == BI_F32) {
        if (!y || ldy < N) return fail(BI_ERR_INVALID_ARG, "%s: null y or ldy < N", fn);
        if (K > 0) {
            if (!x || !w) return fail(BI_ERR_INVALID_ARG, "%s: null x or w", fn);
            if (ldx < K || ldw < (w_layout == BI_W_NK ? K : N))
                return fail(BI_ERR_INVALID_ARG, "%s: ldx or ldw too small", fn);
        }
        if (!aligned(y, 4) || (K > 0 && (!aligned(x, 4) || !aligned(w, 4))))
            return fail(BI_ERR_INVALID_ARG, "%s: pointers not element-aligned", fn);
        cudaError_t why = cudaSuccess;
        if (!current_device_info(&why)) return cuda_fail(why, fn);
        cudaError_t e = launch_gemm_f32(x, ldx, w, ldw, w_layout == BI_W_KN, y, ldy, M, N, K,
                                        reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, fn);
        return BI_OK;
    }
    if (!y) return fail(BI_ERR_INVALID_ARG, "%s: null y", fn);
    if (ldy < N) return fail(BI_ERR_INVALID_ARG, "%s: ldy < N", fn);
    const size_t ysz = y_dtype == BI_F32 ? 4 : 2;
    if (!aligned(y, ysz)) return fail(BI_ERR_INVALID_ARG, "%s: y not element-aligned", fn);
    if (K > 0) {
        if (!x || !w) return fail(BI_ERR_INVALID_ARG, "%s: null x or w", fn);
        if (ldx < K) return fail(BI_ERR_INVALID_ARG, "%s: ldx < K", fn);
        if (w_layout == BI_W_NK && ldw < K)
            return fail(BI_ERR_INVALID_ARG, "%s: ldw < K for layout NK", fn);
        if (w_layout == BI_W_KN && ldw < N)
            return fail(BI_ERR_INVALID_ARG, "%s: ldw < N for layout KN", fn);
        if (!aligned(x, 16) || !aligned(w, 16) || ldx % 8 != 0 || ldw % 8 != 0)
            return fail(BI_ERR_UNSUPPORTED,
                        "%s: x and w must be 16-byte aligned with ldx, ldw multiples of 8 "
                        "(TMA rule)", fn);
    }
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, fn);
    // inside the limit: the invariant schedule; outside it the split-K kernel may be used
    const bool split_ok = !bi_within_batch_invariant_limit(M);
    cudaError_t e = launch_gemm(*dev, x, ldx, w, ldw, w_layout == BI_W_KN, y, ldy,
                                y_dtype == BI_F32, M, N, K, split_ok, in_dtype == BI_F16,
                                g_weight_prefetch.load() != 0,
                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return BI_OK;
}

bi_status rmsnorm_impl(const char* fn, const void* x, int64_t ldx, const void* gamma, void* y,
                       int64_t ldy, int in_dtype, int y_dtype, int64_t rows, int64_t hidden,
                       float eps, bi_stream_t stream) {
    init_limit_from_env();
    if (rows < 0) return fail(BI_ERR_INVALID_ARG, "%s: negative rows", fn);
    if (hidden < 1 || hidden > (int64_t(1) << 20))
        return fail(BI_ERR_INVALID_ARG, "%s: hidden must be in [1, 2^20]", fn);
    if (in_dtype != BI_BF16 && in_dtype != BI_F16 && in_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: in_dtype must be BI_BF16, BI_F16 or BI_F32", fn);
    if (y_dtype != in_dtype && y_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: y_dtype must be in_dtype or BI_F32", fn);
    if (!std::isfinite(eps) || eps < 0.0f)
        return fail(BI_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", fn);
    if (rows == 0) return BI_OK;
    if (!x || !gamma || !y) return fail(BI_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (ldx < hidden || ldy < hidden)
        return fail(BI_ERR_INVALID_ARG, "%s: ldx and ldy must be >= hidden", fn);
    const size_t ysz = y_dtype == BI_F32 ? 4 : 2;
    const size_t xsz = in_dtype == BI_F32 ? 4 : 2;
    if (!aligned(x, xsz) || !aligned(gamma, xsz) || !aligned(y, ysz))
        return fail(BI_ERR_INVALID_ARG, "%s: pointers not element-aligned", fn);
    cudaError_t why = cudaSuccess;
    if (!current_device_info(&why)) return cuda_fail(why, fn);
    if (in_dtype == BI_F32) {
        cudaError_t e = launch_rmsnorm_f32(x, ldx, gamma, y, ldy, rows, hidden, eps,
                                           reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, fn);
        return BI_OK;
    }
    cudaError_t e = launch_rmsnorm(x, ldx, gamma, y, ldy, y_dtype == BI_F32, rows, hidden, eps,
                                   in_dtype == BI_F16, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return BI_OK;
}

}  // namespace

BI_EXPORT bi_status bi_matmul(const void* x, int64_t ldx, const void* w, int64_t ldw,
                              int w_layout, void* y, int64_t ldy, int y_dtype, int64_t M,
                              int64_t N, int64_t K, bi_stream_t stream) {
    if (y_dtype != BI_BF16 && y_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "bi_matmul: y_dtype must be BI_BF16 or BI_F32");
    return matmul_impl("bi_matmul", x, ldx, w, ldw, w_layout, y, ldy, BI_BF16, y_dtype, M, N, K,
                       stream);
}

BI_EXPORT bi_status bi_matmul_ex(const void* x, int64_t ldx, const void* w, int64_t ldw,
                                 int w_layout, void* y, int64_t ldy, int in_dtype, int y_dtype,
                                 int64_t M, int64_t N, int64_t K, bi_stream_t stream) {
    return matmul_impl("bi_matmul_ex", x, ldx, w, ldw, w_layout, y, ldy, in_dtype, y_dtype, M, N,
                       K, stream);
}

// ================================================================ quantized matmul

namespace {
bi_status qmatmul_impl(const char* fn, const void* x, int64_t ldx, const void* wq, int64_t ldwq,
                       const void* scales, int64_t lds, const void* biases, int64_t ldb,
                       int qformat, int group_size, int w_layout, void* y, int64_t ldy,
                       int y_dtype, int64_t M, int64_t N, int64_t K, bi_stream_t stream) {
    init_limit_from_env();
    if (w_layout != BI_W_NK && w_layout != BI_W_KN)
        return fail(BI_ERR_INVALID_ARG, "%s: w_layout must be BI_W_NK or BI_W_KN", fn);
    const bool kn = w_layout == BI_W_KN;
    if (M < 0 || N < 0 || K < 0) return fail(BI_ERR_INVALID_ARG, "%s: negative M/N/K", fn);
    if (M > kI32Max || N > kI32Max || K > kI32Max)
        return fail(BI_ERR_UNSUPPORTED, "%s: M, N, K must be < 2^31", fn);
    if (qformat < BI_Q_MXFP4 || qformat > BI_Q_AFFINE8)
        return fail(BI_ERR_INVALID_ARG, "%s: unknown qformat", fn);
    const bool affine = qformat == BI_Q_AFFINE4 || qformat == BI_Q_AFFINE8;
    const int want_gs = qformat == BI_Q_NVFP4 ? 16 : 32;
    if (affine ? (group_size != 32 && group_size != 64 && group_size != 128)
               : group_size != want_gs)
        return fail(BI_ERR_INVALID_ARG, "%s: group_size must be %s", fn,
                    affine ? "32, 64 or 128" : (want_gs == 16 ? "16" : "32"));
    if (!kn && K % group_size != 0)
        return fail(BI_ERR_INVALID_ARG, "%s: K must be a multiple of group_size", fn);
    if (kn && N % group_size != 0)
        return fail(BI_ERR_INVALID_ARG,
                    "%s: N must be a multiple of group_size (layout KN: groups along N)", fn);
    if (y_dtype != BI_BF16 && y_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "%s: y_dtype must be BI_BF16 or BI_F32", fn);
    if (M == 0 || N == 0) return BI_OK;
    if (!y || ldy < N) return fail(BI_ERR_INVALID_ARG, "%s: null y or ldy < N", fn);
    const size_t ysz = y_dtype == BI_F32 ? 4 : 2;
    if (!aligned(y, ysz)) return fail(BI_ERR_INVALID_ARG, "%s: y not element-aligned", fn);
    if (K > 0) {
        const bool eight = qformat == BI_Q_MXFP8 || qformat == BI_Q_AFFINE8;
        // packed codes and groups run along the quantized dimension: K (layout NK, a row
        // per output column) or N (layout KN, a row per k)
        const int64_t qdim = kn ? N : K;
        const int64_t row_bytes = eight ? qdim : qdim / 2;
        if (!x || !wq || !scales || (affine && !biases))
            return fail(BI_ERR_INVALID_ARG, "%s: null x, wq, scales or biases", fn);
        if (ldx < K || ldwq < row_bytes || lds < qdim / group_size ||
            (affine && ldb < qdim / group_size))
            return fail(BI_ERR_INVALID_ARG, "%s: a row stride is too small", fn);
        if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(wq, 16) || ldwq % 16 != 0)
            return fail(BI_ERR_UNSUPPORTED,
                        "%s: x and wq must be 16-byte aligned, ldx a multiple of 8 and ldwq a "
                        "multiple of 16 bytes (TMA rule)", fn);
        if (affine && (!aligned(scales, 2) || !aligned(biases, 2)))
            return fail(BI_ERR_INVALID_ARG, "%s: scales and biases not element-aligned", fn);
    }
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, fn);
    cudaError_t e =
        kn ? launch_qgemm_kn(*dev, x, ldx, wq, ldwq, scales, lds, biases, ldb, qformat,
                             group_size, y, ldy, y_dtype == BI_F32, M, N, K,
                             g_weight_prefetch.load() != 0, reinterpret_cast<cudaStream_t>(stream))
           : launch_qgemm(*dev, x, ldx, wq, ldwq, scales, lds, biases, ldb, qformat,
                          group_size, y, ldy, y_dtype == BI_F32, M, N, K,
                          g_weight_prefetch.load() != 0, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return BI_OK;
}
}  // namespace

BI_EXPORT bi_status bi_qmatmul(const void* x, int64_t ldx, const void* wq, int64_t ldwq,
                               const void* scales, int64_t lds, const void* biases, int64_t ldb,
                               int qformat, int group_size, void* y, int64_t ldy, int y_dtype,
                               int64_t M, int64_t N, int64_t K, bi_stream_t stream) {
    return qmatmul_impl("bi_qmatmul", x, ldx, wq, ldwq, scales, lds, biases, ldb, qformat,
                        group_size, BI_W_NK, y, ldy, y_dtype, M, N, K, stream);
}

BI_EXPORT bi_status bi_qmatmul_ex(const void* x, int64_t ldx, const void* wq, int64_t ldwq,
                                  const void* scales, int64_t lds, const void* biases,
                                  int64_t ldb, int qformat, int group_size, int w_layout, void* y,
                                  int64_t ldy, int y_dtype, int64_t M, int64_t N, int64_t K,
                                  bi_stream_t stream) {
    return qmatmul_impl("bi_qmatmul_ex", x, ldx, wq, ldwq, scales, lds, biases, ldb, qformat,
                        group_size, w_layout, y, ldy, y_dtype, M, N, K, stream);
}

// ========================================================================= rmsnorm

BI_EXPORT bi_status bi_rmsnorm(const void* x, int64_t ldx, const void* gamma, void* y,
                               int64_t ldy, int y_dtype, int64_t rows, int64_t hidden, float eps,
                               bi_stream_t stream) {
    if (y_dtype != BI_BF16 && y_dtype != BI_F32)
        return fail(BI_ERR_INVALID_ARG, "bi_rmsnorm: y_dtype must be BI_BF16 or BI_F32");
    return rmsnorm_impl("bi_rmsnorm", x, ldx, gamma, y, ldy, BI_BF16, y_dtype, rows, hidden, eps,
                        stream);
}

BI_EXPORT bi_status bi_rmsnorm_ex(const void* x, int64_t ldx, const void* gamma, void* y,
                                  int64_t ldy, int in_dtype, int y_dtype, int64_t rows,
                                  int64_t hidden, float eps, bi_stream_t stream) {
    return rmsnorm_impl("bi_rmsnorm_ex", x, ldx, gamma, y, ldy, in_dtype, y_dtype, rows, hidden,
                        eps, stream);
}

// ======================================================================= attention

namespace {

bi_status check_paged(const char* fn, const PagedArgs& a, int64_t page_size, bool need_cu_q,
                      bool prefill = false) {
    if (a.batch < 0 || a.total_q < 0)
        return fail(BI_ERR_INVALID_ARG, "%s: negative batch or total_q", fn);
    if (a.head_dim != 64 && a.head_dim != 128)
        return fail(BI_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128", fn);
    if (page_size != BI_PAGE_SIZE)
        return fail(BI_ERR_UNSUPPORTED, "%s: page_size must be %d", fn, BI_PAGE_SIZE);
    if (a.hkv < 1 || a.hq < 1 || a.hq % a.hkv != 0)
        return fail(BI_ERR_INVALID_ARG, "%s: num_q_heads must be a positive multiple of "
                                        "num_kv_heads", fn);
    if (a.num_pages < 1 || a.max_pages < 1)
        return fail(BI_ERR_INVALID_ARG, "%s: num_pages and max_pages must be >= 1", fn);
    if (a.num_pages * a.hkv * BI_PAGE_SIZE > kI32Max)
        return fail(BI_ERR_UNSUPPORTED, "%s: cache too large for 32-bit TMA row coordinates", fn);
    if (prefill) {
        if (a.max_q < 1) return fail(BI_ERR_INVALID_ARG, "%s: max_q must be >= 1", fn);
        const int64_t G = a.hq / a.hkv;
        if (G > 128 || 128 % G != 0)
            return fail(BI_ERR_UNSUPPORTED,
                        "%s: num_q_heads/num_kv_heads must divide 128 (128/G tokens per tile)",
                        fn);
    } else {
        if (a.max_q < 1 || a.max_q > BI_ATTN_MAX_Q)
            return fail(BI_ERR_UNSUPPORTED, "%s: max_q must be in [1, %d]", fn, BI_ATTN_MAX_Q);
        if (a.max_q * (a.hq / a.hkv) > BI_ATTN_MAX_ROWS)
            return fail(BI_ERR_UNSUPPORTED,
                        "%s: max_q * (num_q_heads/num_kv_heads) must be <= %d", fn,
                        BI_ATTN_MAX_ROWS);
    }
    if (a.batch > BI_ATTN_MAX_BATCH)
        return fail(BI_ERR_UNSUPPORTED, "%s: batch must be <= %d", fn, BI_ATTN_MAX_BATCH);
    if (a.max_seq_len < 1 || a.max_seq_len > a.max_pages * BI_PAGE_SIZE)
        return fail(BI_ERR_INVALID_ARG, "%s: max_seq_len must be in [1, max_pages*page_size]",
                    fn);
    if (a.batch > 0) {
        if (a.total_q < a.batch || a.total_q > a.batch * a.max_q)
            return fail(BI_ERR_INVALID_ARG, "%s: total_q must be in [batch, batch*max_q]", fn);
        if (a.total_q > kI32Max / (a.hq > a.hkv ? a.hq : a.hkv))
            return fail(BI_ERR_UNSUPPORTED, "%s: total_q too large", fn);
        if (!a.k_cache || !a.v_cache || !a.block_table || !a.seq_lens || (need_cu_q && !a.cu_q))
            return fail(BI_ERR_INVALID_ARG, "%s: null cache / table pointer", fn);
        if (!aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) || !aligned(a.block_table, 4) ||
            !aligned(a.seq_lens, 4) || (a.cu_q && !aligned(a.cu_q, 4)))
            return fail(BI_ERR_UNSUPPORTED, "%s: caches must be 16-byte aligned", fn);
    }
    return BI_OK;
}

bi_status run_attention(const char* fn, const void* q, const PagedArgs& a, int64_t page_size,
                        float scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                        bi_stream_t stream) {
    init_limit_from_env();
    bi_status s = check_paged(fn, a, page_size, a.cu_q != nullptr);
    if (s != BI_OK) return s;
    if (!std::isfinite(scale)) return fail(BI_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    if (a.batch == 0) return BI_OK;
    if (!q || !out || !workspace) return fail(BI_ERR_INVALID_ARG, "%s: null q/out/workspace", fn);
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16) || (lse && !aligned(lse, 4)))
        return fail(BI_ERR_UNSUPPORTED, "%s: q, out and workspace must be 16-byte aligned", fn);
    const size_t need = attn_workspace_bytes(a.total_q, a.hq, a.head_dim, a.max_seq_len);
    if (ws_bytes < need)
        return fail(BI_ERR_INVALID_ARG, "%s: workspace too small (%zu < %zu bytes)", fn, ws_bytes,
                    need);
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, fn);
    // inside the limit (verify width max_q): the fixed chunk length; outside it a chunk
    // length chosen from the call's parallelism
    const int chunk_log2 = attn_chunk_log2(a, ws_bytes, dev->num_sms,
                                           bi_within_batch_invariant_limit(a.max_q) != 0);
    cudaError_t e = launch_attention(*dev, q, a, scale, out, lse, workspace, chunk_log2,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return BI_OK;
}

}  // namespace

BI_EXPORT bi_status bi_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, int64_t num_pages, const int32_t* block_table,
                                 int64_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                                 int64_t batch, int64_t total_q, int64_t num_kv_heads,
                                 int64_t head_dim, int64_t page_size, bi_stream_t stream) {
    init_limit_from_env();
    PagedArgs a{k_cache, v_cache, num_pages, block_table, max_pages, seq_lens, cu_q, batch,
                total_q, BI_ATTN_MAX_Q, int64_t(max_pages) * BI_PAGE_SIZE, num_kv_heads,
                num_kv_heads, head_dim};
    if (batch < 0 || total_q < 0)
        return fail(BI_ERR_INVALID_ARG, "bi_kv_append: negative batch or total_q");
    if (head_dim != 64 && head_dim != 128)
        return fail(BI_ERR_UNSUPPORTED, "bi_kv_append: head_dim must be 64 or 128");
    if (page_size != BI_PAGE_SIZE)
        return fail(BI_ERR_UNSUPPORTED, "bi_kv_append: page_size must be %d", BI_PAGE_SIZE);
    if (num_kv_heads < 1 || num_pages < 1 || max_pages < 1)
        return fail(BI_ERR_INVALID_ARG, "bi_kv_append: num_kv_heads, num_pages, max_pages >= 1");
    if (batch == 0 || total_q == 0) return BI_OK;
    if (total_q < batch && cu_q == nullptr)
        return fail(BI_ERR_INVALID_ARG, "bi_kv_append: total_q < batch without cu_q");
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens || !cu_q)
        return fail(BI_ERR_INVALID_ARG, "bi_kv_append: null pointer");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(BI_ERR_UNSUPPORTED, "bi_kv_append: tensors must be 16-byte aligned");
    if (total_q > kI32Max / num_kv_heads)
        return fail(BI_ERR_UNSUPPORTED, "bi_kv_append: total_q too large");
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, "bi_kv_append: device query");
    cudaError_t e = launch_kv_append(*dev, k_new, v_new, k_cache, v_cache, a,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bi_kv_append: launch");
    return BI_OK;
}

BI_EXPORT size_t bi_attn_workspace_size(int64_t total_q, int64_t num_q_heads, int64_t head_dim,
                                        int64_t max_seq_len) {
    if (total_q < 0 || num_q_heads < 1 || (head_dim != 64 && head_dim != 128) || max_seq_len < 1)
        return 0;
    return attn_workspace_bytes(total_q, num_q_heads, head_dim, max_seq_len);
}

BI_EXPORT bi_status bi_verify_block(const void* q, const void* k_cache, const void* v_cache,
                                    int64_t num_pages, const int32_t* block_table,
                                    int64_t max_pages, const int32_t* seq_lens,
                                    const int32_t* cu_q, int64_t batch, int64_t total_q,
                                    int64_t max_q, int64_t max_seq_len, int64_t num_q_heads,
                                    int64_t num_kv_heads, int64_t head_dim, int64_t page_size,
                                    float scale, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, bi_stream_t stream) {
    if (batch > 0 && !cu_q) return fail(BI_ERR_INVALID_ARG, "bi_verify_block: null cu_q");
    PagedArgs a{k_cache, v_cache, num_pages, block_table, max_pages, seq_lens, cu_q, batch,
                total_q, max_q, max_seq_len, num_q_heads, num_kv_heads, head_dim};
    return run_attention("bi_verify_block", q, a, page_size, scale, out, lse, workspace,
                         workspace_bytes, stream);
}

BI_EXPORT bi_status bi_prefill_attn(const void* q, const void* k_cache, const void* v_cache,
                                    int64_t num_pages, const int32_t* block_table,
                                    int64_t max_pages, const int32_t* seq_lens,
                                    const int32_t* cu_q, int64_t batch, int64_t total_q,
                                    int64_t max_q, int64_t max_seq_len, int64_t num_q_heads,
                                    int64_t num_kv_heads, int64_t head_dim, int64_t page_size,
                                    float scale, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, bi_stream_t stream) {
    const char* fn = "bi_prefill_attn";
    PagedArgs a{k_cache, v_cache, num_pages, block_table, max_pages, seq_lens, cu_q, batch,
                total_q, max_q, max_seq_len, num_q_heads, num_kv_heads, head_dim};
    bi_status s = check_paged(fn, a, page_size, true, true);
    if (s != BI_OK) return s;
    if (!std::isfinite(scale)) return fail(BI_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    if (a.batch == 0) return BI_OK;
    if (!cu_q) return fail(BI_ERR_INVALID_ARG, "%s: null cu_q", fn);
    if (!q || !out || !workspace) return fail(BI_ERR_INVALID_ARG, "%s: null q/out/workspace", fn);
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16) || (lse && !aligned(lse, 4)))
        return fail(BI_ERR_UNSUPPORTED, "%s: q, out and workspace must be 16-byte aligned", fn);
    const size_t need = attn_workspace_bytes(a.total_q, a.hq, a.head_dim, a.max_seq_len);
    if (workspace_bytes < need)
        return fail(BI_ERR_INVALID_ARG, "%s: workspace too small (%zu < %zu bytes)", fn,
                    workspace_bytes, need);
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, fn);
    cudaError_t e = launch_prefill(*dev, q, a, scale, out, lse, workspace,
                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return BI_OK;
}

BI_EXPORT bi_status bi_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                                   int64_t num_pages, const int32_t* block_table,
                                   int64_t max_pages, const int32_t* seq_lens, int64_t batch,
                                   int64_t max_seq_len, int64_t num_q_heads, int64_t num_kv_heads,
                                   int64_t head_dim, int64_t page_size, float scale, void* out,
                                   float* lse, void* workspace, size_t workspace_bytes,
                                   bi_stream_t stream) {
    PagedArgs a{k_cache, v_cache, num_pages, block_table, max_pages, seq_lens, nullptr, batch,
                batch, 1, max_seq_len, num_q_heads, num_kv_heads, head_dim};
    return run_attention("bi_decode_attn", q, a, page_size, scale, out, lse, workspace,
                         workspace_bytes, stream);
}

// ==================================================================== device status

BI_EXPORT bi_status bi_device_status(bi_stream_t stream) {
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, "bi_device_status: device query");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dev->err_word, 0, sizeof word, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "bi_device_status");
    if (word & kErrTimeout)
        return fail(BI_ERR_TIMEOUT, "a bounded device-side wait ran out (error word 0x%x)", word);
    if (word & kErrDeviceArg)
        return fail(BI_ERR_DEVICE_ARG,
                    "a kernel skipped work on an out-of-range device-resident argument "
                    "(error word 0x%x)", word);
    return BI_OK;
}

BI_EXPORT bi_status bi_selftest_set_wait_budget(uint64_t timeout_ns, bi_stream_t stream) {
    if (timeout_ns != 0ull && (timeout_ns < 1000ull || timeout_ns > 10000000000ull))
        return fail(BI_ERR_INVALID_ARG,
                    "bi_selftest_set_wait_budget: timeout_ns must be 0 or in [1e3, 1e10]");
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, "bi_selftest_set_wait_budget: device query");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // stream-ordered: kernels issued on `stream` after this call read the new budget
    const unsigned long long v = timeout_ns;
    cudaError_t e = cudaMemcpyAsync(dev->err_word + 2, &v, sizeof v, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "bi_selftest_set_wait_budget");
    return BI_OK;
}

BI_EXPORT bi_status bi_selftest_wait_timeout(uint64_t timeout_ns, bi_stream_t stream) {
    if (timeout_ns < 1000ull || timeout_ns > 10000000000ull)
        return fail(BI_ERR_INVALID_ARG, "bi_selftest_wait_timeout: timeout_ns out of range");
    cudaError_t why = cudaSuccess;
    const DeviceInfo* dev = current_device_info(&why);
    if (!dev) return cuda_fail(why, "bi_selftest_wait_timeout: device query");
    cudaError_t e = launch_selftest_wait(*dev, timeout_ns, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bi_selftest_wait_timeout: launch");
    return BI_OK;
}
