// attention.cu -- placeholder until the split-KV kernels land.
#include "common.cuh"
#include "launch.h"

namespace bi {

size_t attn_workspace_bytes(int64_t total_q, int64_t hq, int64_t head_dim, int64_t max_seq_len) {
    const int64_t chunks = (max_seq_len + 511) / 512;
    return size_t(total_q) * size_t(hq) * size_t(chunks) * size_t(head_dim + 2) * 4;
}

cudaError_t launch_kv_append(const DeviceInfo&, const void*, const void*, void*, void*,
                             const PagedArgs&, cudaStream_t) {
    return cudaErrorNotYetImplemented;
}

cudaError_t launch_attention(const DeviceInfo&, const void*, const PagedArgs&, float, void*,
                             float*, void*, cudaStream_t) {
    return cudaErrorNotYetImplemented;
}

}  // namespace bi
