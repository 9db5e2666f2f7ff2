// f32path.cu -- batch-invariant matmul and RMSNorm for fp32 inputs (bi_matmul_ex and
// bi_rmsnorm_ex with in_dtype = BI_F32).
//
// Source: "Fix/speculative shape invariance" (ml-explore/mlx PR 4279), the tester's
// comment (dense matmul at M = 4 also diverges for f32 inputs with the limit off); book
// chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Case 6 / The boring rule item 1 (one reduction order at every batch
// size, no split-K, data-parallel RMSNorm rows).
//
// The tensor cores have no full-precision fp32 operand type, so fp32 runs on the CUDA
// cores.  Matmul: every output element is one thread's chain of fmaf over k = 0, 1, ...,
// K-1 in ascending order, starting from +0 -- whatever the tile shape, the element's
// position in it, or M.  Tiles (16 x 32 for M <= 16, else 64 x 64; 256 threads, each
// owning a 1x2 or 4x4 block of outputs) stage 16-wide K chunks of X and W in shared
// memory; they decide only which thread computes an element.  Out-of-range elements read
// as +0 past K only, where every tile shape pads alike.
// RMSNorm: the tree of the 16-bit kernel -- 256 threads, thread t folding the squares of
// its 8-element groups t, t+256, ... in ascending order (fmaf), an xor butterfly per warp,
// a fixed pairwise tree over the 8 warps -- on fp32 elements.
#include "common.cuh"
#include "launch.h"

namespace bi {
namespace {

constexpr int KC = 16;            // K chunk staged per step
constexpr int GEMM_THREADS = 256;  // a 16 x 16 grid of threads

// X [M, K] row-major (ldx); W layout NK: [N, K] (ldw), KN: [K, N] (ldw); Y fp32 (ldy).
template <int TM, int TN, bool KN>
__global__ void __launch_bounds__(GEMM_THREADS)
gemm_f32_kernel(const float* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                int64_t ldw, float* __restrict__ y, int64_t ldy, int M, int N, int K) {
    constexpr int RM = TM / 16, RN = TN / 16;
    __shared__ float xs[KC][TM + 1];
    __shared__ float ws[KC][TN + 1];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = int(blockIdx.y) * TM, n0 = int(blockIdx.x) * TN;
    float acc[RM][RN];
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += KC) {
        // stage X[m0.., k0..k0+15] and W(k0.., n0..) (+0 outside the matrices)
        for (int e = tid; e < TM * KC; e += GEMM_THREADS) {
            const int mm = e / KC, kk = e % KC;
            const int m = m0 + mm, k = k0 + kk;
            xs[kk][mm] = (m < M && k < K) ? x[int64_t(m) * ldx + k] : 0.f;
        }
        for (int e = tid; e < TN * KC; e += GEMM_THREADS) {
            int nn, kk;
            if (KN) {
                kk = e / TN;
                nn = e % TN;
            } else {
                nn = e / KC;
                kk = e % KC;
            }
            const int n = n0 + nn, k = k0 + kk;
            float v = 0.f;
            if (n < N && k < K) v = KN ? w[int64_t(k) * ldw + n] : w[int64_t(n) * ldw + k];
            ws[kk][nn] = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < KC; ++kk) {  // ascending k, one fmaf per element per k
            float a[RM], b[RN];
#pragma unroll
            for (int i = 0; i < RM; ++i) a[i] = xs[kk][ty * RM + i];
#pragma unroll
            for (int j = 0; j < RN; ++j) b[j] = ws[kk][tx * RN + j];
#pragma unroll
            for (int i = 0; i < RM; ++i)
#pragma unroll
                for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < RM; ++i) {
        const int m = m0 + ty * RM + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < RN; ++j) {
            const int n = n0 + tx * RN + j;
            if (n < N) y[int64_t(m) * ldy + n] = acc[i][j];
        }
    }
}

constexpr int RMS_THREADS = 256;

__global__ void __launch_bounds__(RMS_THREADS)
rmsnorm_f32_kernel(const float* __restrict__ x, int64_t ldx, const float* __restrict__ gamma,
                   float* __restrict__ y, int64_t ldy, int H, float eps) {
    __shared__ float warp_sums[RMS_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    const float* xr = x + int64_t(blockIdx.x) * ldx;
    float* yr = y + int64_t(blockIdx.x) * ldy;
    const int groups = (H + 7) / 8;
    float acc = 0.f;
    for (int g = threadIdx.x; g < groups; g += RMS_THREADS)
        for (int i = 0; i < 8; ++i) {
            const int e = g * 8 + i;
            const float v = e < H ? xr[e] : 0.f;
            acc = fmaf(v, v, acc);
        }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = acc;
    __syncthreads();
    const float s01 = warp_sums[0] + warp_sums[1];
    const float s23 = warp_sums[2] + warp_sums[3];
    const float s45 = warp_sums[4] + warp_sums[5];
    const float s67 = warp_sums[6] + warp_sums[7];
    const float ss = (s01 + s23) + (s45 + s67);
    const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
    for (int e = threadIdx.x; e < H; e += RMS_THREADS) yr[e] = (xr[e] * inv) * gamma[e];
}

}  // namespace

cudaError_t launch_gemm_f32(const void* x, int64_t ldx, const void* w, int64_t ldw, bool w_kn,
                            void* y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                            cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0)
        return cudaMemset2DAsync(y, size_t(ldy) * 4, 0, size_t(N) * 4, size_t(M), stream);
    auto xf = static_cast<const float*>(x);
    auto wf = static_cast<const float*>(w);
    auto yf = static_cast<float*>(y);
    const dim3 block(GEMM_THREADS);
    if (M <= 16) {
        const dim3 grid(unsigned((N + 31) / 32), unsigned((M + 15) / 16));
        return w_kn ? launch_pdl(gemm_f32_kernel<16, 32, true>, grid, block, 0, stream, xf, ldx, wf,
                                 ldw, yf, ldy, int(M), int(N), int(K))
                    : launch_pdl(gemm_f32_kernel<16, 32, false>, grid, block, 0, stream, xf, ldx,
                                 wf, ldw, yf, ldy, int(M), int(N), int(K));
    }
    const int64_t gy = (M + 63) / 64;
    if (gy > 65535) return cudaErrorNotSupported;
    const dim3 grid(unsigned((N + 63) / 64), unsigned(gy));
    return w_kn ? launch_pdl(gemm_f32_kernel<64, 64, true>, grid, block, 0, stream, xf, ldx, wf, ldw,
                             yf, ldy, int(M), int(N), int(K))
                : launch_pdl(gemm_f32_kernel<64, 64, false>, grid, block, 0, stream, xf, ldx, wf,
                             ldw, yf, ldy, int(M), int(N), int(K));
}

cudaError_t launch_rmsnorm_f32(const void* x, int64_t ldx, const void* gamma, void* y,
                               int64_t ldy, int64_t rows, int64_t hidden, float eps,
                               cudaStream_t stream) {
    const int64_t kMaxGrid = 0x7fffffff;
    for (int64_t r0 = 0; r0 < rows; r0 += kMaxGrid) {
        const int64_t n = rows - r0 < kMaxGrid ? rows - r0 : kMaxGrid;
        cudaError_t e = launch_pdl(rmsnorm_f32_kernel, dim3(unsigned(n)), dim3(RMS_THREADS), 0,
                                   stream, static_cast<const float*>(x) + r0 * ldx, ldx,
                                   static_cast<const float*>(gamma),
                                   static_cast<float*>(y) + r0 * ldy, ldy, int(hidden), eps);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace bi
