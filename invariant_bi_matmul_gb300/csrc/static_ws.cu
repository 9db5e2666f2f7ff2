// static_ws.cu -- bi_verify_block for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code that
// runs while a CUDA graph is being recorded or replayed by someone else, allocator-free
// runtimes that hand the library only the tensors they own, or real-time paths where a
// device allocation (and the implicit synchronisation it may cause) is not allowed.  For
// them this file keeps the split-KV workspace in a fixed, file-scope device array and
// forwards to the ordinary bi_verify_block with that array as the workspace.
//
// The array is BI_STATIC_WS_BYTES (32 MiB) and lives on every GPU that loads the library
// until the process exits.  All calls share it and it keeps the last call's contents:
// nothing in it has to start at zero (every partial a call reads is written earlier in
// the same call), but two calls whose kernels overlap on the GPU -- on different streams,
// or from different threads -- race on it and may both return wrong results.
#include <cstdio>
#include <mutex>

#include "bi.h"
#include "launch.h"

namespace bi {

// Defined in api.cu: sets the thread-local message bi_last_error_message() returns.
void set_last_error_message(const char* msg);

namespace {

// The scratch.  In host code this name is a host-side stand-in, not a device address:
// only the pointer obtained from cudaGetSymbolAddress (per device) is passed to kernels.
static __device__ __align__(256) unsigned char g_static_workspace[BI_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device (the
// first call on a device does this set-up).  Returns nullptr and sets `why` on failure.
void* scratch_on_current_device(cudaError_t* why) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess || !p) {
            *why = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
        g_ws_addr[dev] = p;
    }
    return g_ws_addr[dev];
}

}  // namespace
}  // namespace bi

extern "C" __attribute__((visibility("default"))) bi_status bi_verify_block_static_ws(
    const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
    const int32_t* block_table, int64_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
    int64_t batch, int64_t total_q, int64_t max_q, int64_t max_seq_len, int64_t num_q_heads,
    int64_t num_kv_heads, int64_t head_dim, int64_t page_size, float scale, void* out,
    float* lse, bi_stream_t stream) {
    const size_t need = bi_attn_workspace_size(total_q, num_q_heads, head_dim, max_seq_len);
    if (batch > 0 && need > size_t(BI_STATIC_WS_BYTES)) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "bi_verify_block_static_ws: this block needs %zu bytes of workspace, the "
                 "static scratch holds %zu; call bi_verify_block with your own workspace",
                 need, size_t(BI_STATIC_WS_BYTES));
        bi::set_last_error_message(msg);
        return BI_ERR_UNSUPPORTED;
    }
    cudaError_t why = cudaSuccess;
    void* ws = batch > 0 ? bi::scratch_on_current_device(&why) : nullptr;
    if (batch > 0 && !ws) {
        char msg[256];
        snprintf(msg, sizeof msg, "bi_verify_block_static_ws: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(why));
        bi::set_last_error_message(msg);
        return BI_ERR_CUDA;
    }
    // The workspace size passed on is the block's own need, not the scratch's size: outside
    // the batch-invariant limit the chunk length is chosen among those whose partials fit
    // the workspace, so this gives the choice (and the bits) of bi_verify_block called with
    // exactly bi_attn_workspace_size() bytes.
    return bi_verify_block(q, k_cache, v_cache, num_pages, block_table, max_pages, seq_lens, cu_q,
                           batch, total_q, max_q, max_seq_len, num_q_heads, num_kv_heads,
                           head_dim, page_size, scale, out, lse, ws, need, stream);
}
