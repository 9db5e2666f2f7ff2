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
// K-1 in ascending order, starting from +0 (no padded steps past K) -- whatever the tile
// shape, the element's position in it, or M.  Tiles decide only which thread computes an
// element: for M <= 16, 16 x 32 tiles of 1 x 2 outputs per thread over 64-wide K chunks;
// else 128 x 128 tiles of 8 x 8 outputs per thread (64 x 64 of 4 x 4 when the larger tiles
// would leave SMs idle) over 8-wide K chunks, the next chunk loaded into registers while
// the current one is multiplied out of shared memory.
// RMSNorm: the tree of the 16-bit kernel -- 256 threads, thread t folding the squares of
// its 8-element groups t, t+256, ... in ascending order (fmaf), an xor butterfly per warp,
// a fixed pairwise tree over the 8 warps -- on fp32 elements.
#include "common.cuh"
#include "launch.h"

namespace bi {
namespace {

constexpr int GEMM_THREADS = 256;  // a 16 x 16 grid of threads

// X [M, K] row-major (ldx); W layout NK: [N, K] (ldw), KN: [K, N] (ldw); Y fp32 (ldy).
template <int TM, int TN, int KC, bool KN>
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
        const int kn = K - k0 < KC ? K - k0 : KC;  // no steps past K
#pragma unroll 16
        for (int kk = 0; kk < kn; ++kk) {  // ascending k, one fmaf per element per k
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

// BB x BB tile (BB = 128 or 64), 256 threads of R x R outputs (R = BB / 16), 8-wide K
// chunks: chunk c+1 comes from global memory into registers while chunk c is multiplied
// out of shared memory (two shared buffers, one barrier per chunk).  vec: every row of X
// (and of W) starts on a 16-byte boundary and K (N for KN) is a multiple of 4, so vector
// loads never straddle the matrix edge.
constexpr int BKB = 8, BPAD = 4;

template <int BB, bool KN>
__global__ void __launch_bounds__(GEMM_THREADS)
gemm_f32_big_kernel(const float* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                    int64_t ldw, float* __restrict__ y, int64_t ldy, int M, int N, int K,
                    int vec) {
    constexpr int R = BB / 16;          // outputs per thread along each dimension
    constexpr int E = BB * BKB / GEMM_THREADS;  // chunk elements each thread loads: 4 or 2
    __shared__ __align__(16) float as[2][BKB][BB + BPAD];
    __shared__ __align__(16) float bs[2][BKB][BB + BPAD];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = int(blockIdx.y) * BB, n0 = int(blockIdx.x) * BB;
    // this thread's E consecutive elements of the X chunk (and of the W chunk):
    // NK / X: row tid/(8/E), k (tid%(8/E))*E..; KN: k tid/(BB/E), n (tid%(BB/E))*E..
    const int lr = tid / (BKB / E), lk = (tid % (BKB / E)) * E;
    const int kr = tid / (BB / E), kc = (tid % (BB / E)) * E;
    float ra[E], rb[E];
    auto vload = [&](const float* p, float (&r)[E]) {
        if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4*>(p);
            r[0] = v.x; r[1 % E] = v.y; r[2 % E] = v.z; r[3 % E] = v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(p);
            r[0] = v.x; r[1 % E] = v.y;
        }
    };
    auto load = [&](int k0) {
        const int m = m0 + lr;
        if (vec) {
            if (m < M && k0 + lk < K) {
                vload(x + int64_t(m) * ldx + k0 + lk, ra);
            } else {
#pragma unroll
                for (int i = 0; i < E; ++i) ra[i] = 0.f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i)
                ra[i] = (m < M && k0 + lk + i < K) ? x[int64_t(m) * ldx + k0 + lk + i] : 0.f;
        }
        if (KN) {
            const int k = k0 + kr, n = n0 + kc;
            if (vec) {
                if (k < K && n < N) {
                    vload(w + int64_t(k) * ldw + n, rb);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i) rb[i] = 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < E; ++i)
                    rb[i] = (k < K && n + i < N) ? w[int64_t(k) * ldw + n + i] : 0.f;
            }
        } else {
            const int n = n0 + lr;
            if (vec) {
                if (n < N && k0 + lk < K) {
                    vload(w + int64_t(n) * ldw + k0 + lk, rb);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i) rb[i] = 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < E; ++i)
                    rb[i] = (n < N && k0 + lk + i < K) ? w[int64_t(n) * ldw + k0 + lk + i] : 0.f;
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < E; ++i) as[buf][lk + i][lr] = ra[i];
        if (KN) {
#pragma unroll
            for (int i = 0; i < E; ++i) bs[buf][kr][kc + i] = rb[i];
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) bs[buf][lk + i][lr] = rb[i];
        }
    };
    float acc[R][R];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < R; ++j) acc[i][j] = 0.f;
    load(0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += BKB) {
        const bool more = k0 + BKB < K;
        if (more) load(k0 + BKB);  // in flight while this chunk is multiplied
        const int kn = K - k0 < BKB ? K - k0 : BKB;  // no steps past K
#pragma unroll
        for (int kk = 0; kk < BKB; ++kk) {  // ascending k, one fmaf per element per k
            if (kk < kn) {
                float a[R], b[R];
#pragma unroll
                for (int q = 0; q < R; q += 4) {
                    const float4 av = *reinterpret_cast<const float4*>(&as[buf][kk][ty * R + q]);
                    const float4 bv = *reinterpret_cast<const float4*>(&bs[buf][kk][tx * R + q]);
                    a[q] = av.x; a[q + 1] = av.y; a[q + 2] = av.z; a[q + 3] = av.w;
                    b[q] = bv.x; b[q + 1] = bv.y; b[q + 2] = bv.z; b[q + 3] = bv.w;
                }
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int j = 0; j < R; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }
        if (more) store(buf ^ 1);  // the other buffer: last read before the previous barrier
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int m = m0 + ty * R + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int n = n0 + tx * R + j;
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
        return w_kn ? launch_pdl(gemm_f32_kernel<16, 32, 64, true>, grid, block, 0, stream, xf, ldx,
                                 wf, ldw, yf, ldy, int(M), int(N), int(K))
                    : launch_pdl(gemm_f32_kernel<16, 32, 64, false>, grid, block, 0, stream, xf,
                                 ldx, wf, ldw, yf, ldy, int(M), int(N), int(K));
    }
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const int vec = al16(x) && al16(w) && ldx % 4 == 0 && ldw % 4 == 0 && K % 4 == 0 &&
                    (!w_kn || N % 4 == 0);
    // 128 x 128 tiles when they give every SM a tile, else 64 x 64 (four times as many)
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool big = ((M + 127) / 128) * ((N + 127) / 128) >= sms;
    const int bb = big ? 128 : 64;
    const int64_t gy = (M + bb - 1) / bb;
    if (gy > 65535) return cudaErrorNotSupported;
    const dim3 grid(unsigned((N + bb - 1) / bb), unsigned(gy));
    if (big)
        return w_kn ? launch_pdl(gemm_f32_big_kernel<128, true>, grid, block, 0, stream, xf, ldx,
                                 wf, ldw, yf, ldy, int(M), int(N), int(K), vec)
                    : launch_pdl(gemm_f32_big_kernel<128, false>, grid, block, 0, stream, xf, ldx,
                                 wf, ldw, yf, ldy, int(M), int(N), int(K), vec);
    return w_kn ? launch_pdl(gemm_f32_big_kernel<64, true>, grid, block, 0, stream, xf, ldx, wf,
                             ldw, yf, ldy, int(M), int(N), int(K), vec)
                : launch_pdl(gemm_f32_big_kernel<64, false>, grid, block, 0, stream, xf, ldx, wf,
                             ldw, yf, ldy, int(M), int(N), int(K), vec);
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
