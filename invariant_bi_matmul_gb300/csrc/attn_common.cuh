// attn_common.cuh -- what the split-KV attention kernels (decode / verify in attention.cu,
// chunked prefill in prefill.cu) share: the page and invariant chunk lengths, the lazy
// rescale threshold, the swizzled tile addressing and the per-sequence block geometry.
// The per-query reduction both kernels implement is described at the top of
// attention.cu; prefill.cu reproduces it row by row.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "bi.h"

namespace bi {

constexpr int PAGE = 64;
constexpr int CHUNK_LOG2 = 9;  // the invariant chunk length: 512 keys
constexpr int CHUNK = 1 << CHUNK_LOG2;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the row max grows by > 2^8
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x by the hardware's approximation (PTX ex2.approx.ftz.f32: at most 2 ulp from 2^x;
// results below 2^-126 flush to +0; 2^-inf = +0).  The softmax of every split-KV kernel
// takes P and the rescale factors from this one function, so they agree bit for bit.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// byte offset of (row, 16-byte chunk) in a 128-byte-swizzled box (the TMA SWIZZLE_128B
// pattern: chunk index XOR row mod 8)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return uint32_t(row) * 128u + (uint32_t((chunk ^ (row & 7)) & 7) << 4);
}

// sequence b's block: length L (new tokens included), block width qb, first token t0
struct SeqInfo {
    int L, qb, t0;
};

__device__ __forceinline__ SeqInfo seq_info(const int32_t* seq_lens, const int32_t* cu_q, int b) {
    SeqInfo s;
    s.L = seq_lens[b];
    if (cu_q) {
        s.t0 = cu_q[b];
        s.qb = cu_q[b + 1] - s.t0;
    } else {
        s.t0 = b;
        s.qb = 1;
    }
    return s;
}

__device__ __forceinline__ bool seq_ok(const SeqInfo& s, int max_q, int max_seq_len, int total_q) {
    return s.L >= 1 && s.L <= max_seq_len && s.qb >= 1 && s.qb <= max_q && s.qb <= s.L &&
           s.t0 >= 0 && s.t0 + s.qb <= total_q;
}

}  // namespace bi
