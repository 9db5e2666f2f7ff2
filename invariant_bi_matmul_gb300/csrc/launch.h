// launch.h -- host-side launchers of the libbi kernels (internal; the public surface is
// include/bi.h).  Arguments are already validated by api.cu when these are called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace bi {

// Bits of the per-device error word (the host maps them to bi_status codes).
enum : unsigned int {
    kErrTimeout = 1u,    // a bounded wait ran out
    kErrDeviceArg = 2u,  // a device-resident argument was out of range; work skipped
};

// Launches `kernel` with programmatic dependent launch allowed: the next kernel in the
// stream may be scheduled as soon as every CTA of this one has started (each kernel
// triggers its dependents early), and each kernel waits (griddepcontrol.wait) for the
// previous grid to complete and flush before it touches global memory.  Only launch
// latency and prologues overlap; completion order and memory visibility are unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl for a kernel launched in clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    unsigned int* err_word = nullptr;  // device address of this device's error word
};

// Current device's cached properties and error-word address (nullptr on failure).
const DeviceInfo* current_device_info(cudaError_t* why);

// ---------------------------------------------------------------- RMSNorm (rmsnorm.cu)
cudaError_t launch_rmsnorm(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                           bool y_f32, int64_t rows, int64_t hidden, float eps, bool f16,
                           cudaStream_t stream);

// ------------------------------------------------------------------- GEMM (gemm.cu)
// Returns cudaErrorNotSupported when a TMA descriptor cannot be encoded.  w_early: W
// may be read before the previous grid in the stream has finished (it does not write W).
cudaError_t launch_gemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* w,
                        int64_t ldw, bool w_kn, void* y, int64_t ldy, bool y_f32, int64_t M,
                        int64_t N, int64_t K, bool split_ok, bool f16, bool w_early,
                        cudaStream_t stream);
int gemm_tile_n();

// Quantized W (gemm.cu): bf16 X times W decoded from packed codes (format 0 mxfp4,
// 1 nvfp4, 2 mxfp8, 3 affine 4-bit, 4 affine 8-bit) with the invariant GEMM's
// instruction sequence.  Returns cudaErrorNotSupported when a descriptor cannot be made.
cudaError_t launch_qgemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* wq,
                         int64_t ldq, const void* scales, int64_t lds, const void* biases,
                         int64_t ldb, int fmt, int gs, void* y, int64_t ldy, bool y_f32,
                         int64_t M, int64_t N, int64_t K, bool w_early, cudaStream_t stream);

// The same for W in the natural layout: codes [K, N] quantized along N (one scale per
// group of gs consecutive columns of a row).
cudaError_t launch_qgemm_kn(const DeviceInfo& dev, const void* x, int64_t ldx, const void* wq,
                            int64_t ldq, const void* scales, int64_t lds, const void* biases,
                            int64_t ldb, int fmt, int gs, void* y, int64_t ldy, bool y_f32,
                            int64_t M, int64_t N, int64_t K, bool w_early, cudaStream_t stream);

// fp32 inputs (f32path.cu): CUDA-core matmul, one ascending fmaf chain per element, and
// RMSNorm with the 16-bit kernel's tree.  y fp32.
cudaError_t launch_gemm_f32(const void* x, int64_t ldx, const void* w, int64_t ldw, bool w_kn,
                            void* y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                            cudaStream_t stream);
cudaError_t launch_rmsnorm_f32(const void* x, int64_t ldx, const void* gamma, void* y,
                               int64_t ldy, int64_t rows, int64_t hidden, float eps,
                               cudaStream_t stream);

// How a GEMM launch is scheduled: X rows staged per K-block, instruction tiles per CTA
// tile, shared-memory ring depth, CTA tiles -- none of which changes what an element
// computes -- and, only when split_ok (a call outside the batch-invariant limit), the
// split-K factor, which does.
struct GemmSchedule {
    int a_rows = 128;
    int nsub = 1;
    int kbs = 1;
    int blocked = 0;
    int stages = 0;
    int ring_bytes = 0;
    int splits = 1;        // CTAs (one cluster) per output tile, each over a K range
    int kb_per_split = 0;  // 64-wide K-blocks per split
    int kn_wide = 0;       // layout KN: W staged in 64-column atoms
    int64_t tiles = 0;
};
GemmSchedule gemm_schedule(int64_t M, int64_t N, int64_t K, bool w_kn, int num_sms,
                           bool split_ok);

// ------------------------------------------------------------ attention (attention.cu)
struct PagedArgs {
    const void* k_cache;
    const void* v_cache;
    int64_t num_pages;
    const int32_t* block_table;
    int64_t max_pages;
    const int32_t* seq_lens;
    const int32_t* cu_q;  // nullptr: one token per sequence (decode)
    int64_t batch;
    int64_t total_q;
    int64_t max_q;
    int64_t max_seq_len;
    int64_t hq;
    int64_t hkv;
    int64_t head_dim;
};

cudaError_t launch_kv_append(const DeviceInfo& dev, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, const PagedArgs& a,
                             cudaStream_t stream);

size_t attn_workspace_bytes(int64_t total_q, int64_t hq, int64_t head_dim, int64_t max_seq_len);

// The split-KV chunk length (log2 of keys per work item) of a call: the fixed invariant
// length when `invariant`, else the length a cost model picks from the call's sizes,
// the SM count and the workspace.
int attn_chunk_log2(const PagedArgs& a, size_t ws_bytes, int num_sms, bool invariant);

cudaError_t launch_attention(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                             float scale, void* out, float* lse, void* workspace,
                             int chunk_log2, cudaStream_t stream);

// The log-sum-exp merge of the chunk partials in `workspace` (as the split-KV kernels
// leave them for chunk length 2^chunk_log2) into out (and lse).  With `cnt` (the item
// counters the decode / verify partial kernel increments) each row waits for its own
// (sequence, KV head)'s items and the merge may overlap the partial kernel; with nullptr
// it waits for the whole previous grid.  Timeouts are latched in `err`.
cudaError_t launch_attn_merge(const PagedArgs& a, void* workspace, int chunk_log2, void* out,
                              float* lse, const unsigned int* cnt, unsigned int* err,
                              cudaStream_t stream);

// Chunked prefill (prefill.cu): blocks of any width, each query reduced exactly as the
// decode / verify kernels reduce it (invariant chunk length), then the same merge.
cudaError_t launch_prefill(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                           float scale, void* out, float* lse, void* workspace,
                           cudaStream_t stream);

cudaError_t launch_selftest_wait(const DeviceInfo& dev, unsigned long long timeout_ns,
                                 cudaStream_t stream);

}  // namespace bi
