// rmsnorm.cu -- batch-invariant RMSNorm.
//
// Book chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Case 4 (RMSNorm definition; a tree that changes with the batch
// changes every element) and Case 6 strategy table, RMSNorm row: keep the reduction
// data-parallel, one row per core, and accept idle SMs at batch 1.
//
// One CTA of 256 threads owns one row.  The row is cut into 8-element groups; thread t
// owns groups t, t+256, t+512, ... and folds their squares in ascending element order
// (fp32).  The 256 per-thread sums are combined by an xor-butterfly inside each warp
// (every lane ends with the same bits) and then by a fixed pairwise tree over the 8
// warps.  The whole tree is a function of H alone, so a row's bits never depend on the
// number of rows in the launch, on the row's index, or on the memory alignment (the
// 128-bit and scalar load paths do the same arithmetic).
#include "common.cuh"
#include "launch.h"

namespace bi {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxGroupsInRegs = 8;  // H <= 8 * 256 * 8 = 16384 keeps x in registers

// One 8-element group as packed bf16 (elements past H read as +0, whose square adds an
// exact +0: the same as skipping them).
__device__ __forceinline__ uint4 load_group_raw(const __nv_bfloat16* __restrict__ row, int64_t g,
                                                int H, bool vec) {
    const int64_t e0 = g * 8;
    if (vec && e0 + 8 <= H) return __ldg(reinterpret_cast<const uint4*>(row + e0));
    uint16_t h[8];
    const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = (e0 + i < H) ? r16[e0 + i] : uint16_t(0);
    return make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                      h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
}

// Eight 16-bit values widened to fp32 (exact): bf16, or IEEE binary16 when f16.
__device__ __forceinline__ void unpack_group(const uint4& raw, float (&v)[8], bool f16) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (f16) {
            v[2 * i] = widen16(uint16_t(w[i] & 0xffffu), true);
            v[2 * i + 1] = widen16(uint16_t(w[i] >> 16), true);
        } else {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

__device__ __forceinline__ void load_group(const __nv_bfloat16* __restrict__ row, int64_t g,
                                           int H, bool vec, float (&v)[8], bool f16) {
    unpack_group(load_group_raw(row, g, H, vec), v, f16);
}

template <bool F32OUT>
__device__ __forceinline__ void store_group(void* __restrict__ yrow, int64_t g, int H, bool vec,
                                            const float (&o)[8], bool f16) {
    const int64_t e0 = g * 8;
    if (vec && e0 + 8 <= H) {
        if (F32OUT) {
            float4* p = reinterpret_cast<float4*>(static_cast<float*>(yrow) + e0);
            p[0] = make_float4(o[0], o[1], o[2], o[3]);
            p[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
            uint4 raw;
            raw.x = pack16x2(o[0], o[1], f16);
            raw.y = pack16x2(o[2], o[3], f16);
            raw.z = pack16x2(o[4], o[5], f16);
            raw.w = pack16x2(o[6], o[7], f16);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(yrow) + e0) = raw;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (e0 + i < H) {
                if (F32OUT)
                    static_cast<float*>(yrow)[e0 + i] = o[i];
                else
                    static_cast<uint16_t*>(yrow)[e0 + i] = round16(o[i], f16);
            }
        }
    }
}

// MAXJ > 0: the rows stay in registers (packed bf16) between the two passes
// (H <= 8*256*MAXJ); a CTA takes ROWS consecutive rows, each reduced exactly as if it
// were alone.  MAXJ == 0: one row per CTA, and the second pass reads it again (very wide
// rows).  MAXJ and ROWS only bound loops; the per-thread order (ascending group,
// ascending element), the butterfly and the warp tree of a row -- and therefore its
// bits -- are the same for every MAXJ that fits H and every ROWS.
template <int MAXJ, bool F32OUT, int ROWS>
__global__ void __launch_bounds__(kThreads)
rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
               const __nv_bfloat16* __restrict__ gamma, void* __restrict__ y, int64_t ldy,
               int64_t rows, int H, float eps, int vec, int f16) {
    __shared__ float warp_sums[ROWS][kWarps];
    pdl_wait();
    pdl_trigger();
    const int64_t row0 = int64_t(blockIdx.x) * ROWS;
    const int64_t ngroups = (H + 7) / 8;
    const int t = threadIdx.x;
    const bool v16 = vec != 0;
    const bool h16 = f16 != 0;  // x, gamma (and a 16-bit y) are binary16 instead of bf16
    constexpr int J = MAXJ > 0 ? MAXJ : 1;

    float acc[ROWS];
    uint4 xs[ROWS][J], gs[J];
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) acc[rr] = 0.0f;
    if (MAXJ > 0) {
        // the rows and gamma are all requested before any arithmetic: gamma's (L2) round
        // trip overlaps the rows' instead of following the reduction
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const __nv_bfloat16* __restrict__ xr = x + (row0 + rr) * ldx;
            const bool live = row0 + rr < rows;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int64_t g = t + static_cast<int64_t>(j) * kThreads;
                xs[rr][j] = (live && g < ngroups) ? load_group_raw(xr, g, H, v16)
                                                  : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int64_t g = t + static_cast<int64_t>(j) * kThreads;
            gs[j] = (g < ngroups) ? load_group_raw(gamma, g, H, v16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int64_t g = t + static_cast<int64_t>(j) * kThreads;
                if (g < ngroups) {
                    float v[8];
                    unpack_group(xs[rr][j], v, h16);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[rr] = fmaf(v[i], v[i], acc[rr]);
                }
            }
        }
    } else {
        const __nv_bfloat16* __restrict__ xr = x + row0 * ldx;
        for (int64_t g = t; g < ngroups; g += kThreads) {
            float v[8];
            load_group(xr, g, H, v16, v, h16);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[0] = fmaf(v[i], v[i], acc[0]);
        }
    }

    // warp butterfly: every lane ends with identical bits (each step is a+b on a pair)
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            acc[rr] += __shfl_xor_sync(0xffffffffu, acc[rr], off);
        if ((t & 31) == 0) warp_sums[rr][t >> 5] = acc[rr];
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
        const int64_t row = row0 + rr;
        if (row >= rows) break;
        // fixed pairwise tree over the 8 warp partials, evaluated by every thread
        const float s01 = warp_sums[rr][0] + warp_sums[rr][1];
        const float s23 = warp_sums[rr][2] + warp_sums[rr][3];
        const float s45 = warp_sums[rr][4] + warp_sums[rr][5];
        const float s67 = warp_sums[rr][6] + warp_sums[rr][7];
        const float ss = (s01 + s23) + (s45 + s67);
        const float inv = rsqrtf(ss / static_cast<float>(H) + eps);

        void* yrow = F32OUT ? static_cast<void*>(static_cast<float*>(y) + row * ldy)
                            : static_cast<void*>(static_cast<__nv_bfloat16*>(y) + row * ldy);
        if (MAXJ > 0) {
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int64_t g = t + static_cast<int64_t>(j) * kThreads;
                if (g < ngroups) {
                    float v[8], gm[8], o[8];
                    unpack_group(xs[rr][j], v, h16);
                    unpack_group(gs[j], gm, h16);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = (v[i] * inv) * gm[i];
                    store_group<F32OUT>(yrow, g, H, v16, o, h16);
                }
            }
        } else {
            const __nv_bfloat16* __restrict__ xr = x + row * ldx;
            for (int64_t g = t; g < ngroups; g += kThreads) {
                float v[8], gm[8], o[8];
                load_group(xr, g, H, v16, v, h16);
                load_group(gamma, g, H, v16, gm, h16);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = (v[i] * inv) * gm[i];
                store_group<F32OUT>(yrow, g, H, v16, o, h16);
            }
        }
    }
}

template <int MAXJ, int ROWS>
cudaError_t launch_impl(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                        bool y_f32, int64_t rows, int H, float eps, int vec, int f16,
                        cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((rows + ROWS - 1) / ROWS)), block(kThreads);
    auto xb = static_cast<const __nv_bfloat16*>(x);
    auto gb = static_cast<const __nv_bfloat16*>(gamma);
    if (y_f32)
        return launch_pdl(rmsnorm_kernel<MAXJ, true, ROWS>, grid, block, 0, s, xb, ldx, gb, y,
                          ldy, rows, H, eps, vec, f16);
    return launch_pdl(rmsnorm_kernel<MAXJ, false, ROWS>, grid, block, 0, s, xb, ldx, gb, y, ldy,
                      rows, H, eps, vec, f16);
}

}  // namespace

cudaError_t launch_rmsnorm(const void* x, int64_t ldx, const void* gamma, void* y, int64_t ldy,
                           bool y_f32, int64_t rows, int64_t hidden, float eps, bool f16,
                           cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int H = static_cast<int>(hidden);
    const int h16 = f16 ? 1 : 0;
    const size_t ysz = y_f32 ? 4 : 2;
    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ldx % 8 == 0) &&
                     (reinterpret_cast<uintptr_t>(gamma) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(y) % 16 == 0) && ((ldy * ysz) % 16 == 0);
    // rows beyond 2^31-1 CTAs are launched in slices; each CTA still owns one row.
    const int64_t kMaxGrid = 0x7fffffff;
    for (int64_t r0 = 0; r0 < rows; r0 += kMaxGrid) {
        const int64_t n = rows - r0 < kMaxGrid ? rows - r0 : kMaxGrid;
        const void* xs = static_cast<const __nv_bfloat16*>(x) + r0 * ldx;
        void* ys = y_f32 ? static_cast<void*>(static_cast<float*>(y) + r0 * ldy)
                         : static_cast<void*>(static_cast<__nv_bfloat16*>(y) + r0 * ldy);
        const int64_t groups_per_thread = ((H + 7) / 8 + kThreads - 1) / kThreads;
        cudaError_t e;
        // one row per CTA: short CTAs drain the last wave quickly, and at 48 registers
        // five CTAs share an SM (two rows per CTA kept 2x the bytes per thread in flight
        // but measured slower: 13.5 vs 12.6 us at 2048 x 8192)
#define BI_RMS_ARGS xs, ldx, gamma, ys, ldy, y_f32, n, H, eps, vec, h16, stream
        if (groups_per_thread <= 1)
            e = launch_impl<1, 1>(BI_RMS_ARGS);
        else if (groups_per_thread <= 2)
            e = launch_impl<2, 1>(BI_RMS_ARGS);
        else if (groups_per_thread <= 4)
            e = launch_impl<4, 1>(BI_RMS_ARGS);
        else if (groups_per_thread <= kMaxGroupsInRegs)
            e = launch_impl<kMaxGroupsInRegs, 1>(BI_RMS_ARGS);
        else
            e = launch_impl<0, 1>(BI_RMS_ARGS);
#undef BI_RMS_ARGS
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace bi
