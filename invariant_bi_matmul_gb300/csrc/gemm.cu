// gemm.cu -- batch-invariant bf16 GEMM on the 5th-generation tensor cores (tcgen05).
//
// Sources: book chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Case 3 (a K tile picked from the batch size changes row 0) and the
// Case 6 strategy table, Matmul row (one compiled configuration for all shapes, no
// Split-K, no switch to a narrower instruction for small M); "Fix/speculative shape
// invariance" (ml-explore/mlx PR 4279), Problem (GEMV vs gemv_wide vs GEMM chosen by the
// row count is the defect), Changes (rows stay parallel, each with the canonical
// reduction) and the review thread (both B orientations must be covered).
//
// What decides the bits of Y[m, n] -- identical for every M:
//   * the instruction tcgen05.mma.cta_group::1.kind::f16 of shape 128 x 32 x 16 (bf16 in,
//     fp32 accumulator in tensor memory), always with token row m at lane m % 128 of
//     M-tile m / 128 and column n in the 32-wide instruction tile n / 32;
//   * the K order: 64-wide K-blocks in ascending order, and inside a block the four
//     16-wide steps in ascending order, the first one overwriting the accumulator;
//   * the epilogue: fp32 -> bf16 round-to-nearest-even (or fp32 as is).
// What follows M (scheduling only; never an element's instruction sequence):
//   * a_rows: how many X rows are staged per K-block (M rounded up to 8, at most 128).
//     The MMA always reads 128 rows; rows past a_rows read whatever lies in shared
//     memory after the staged rows and land in tensor-memory lanes that are never
//     stored, so no real row depends on them;
//   * nsub: how many adjacent 32-wide instruction tiles one CTA covers with the X block
//     it staged (1 for small M to spread W over every SM, up to 8 for large M to stop
//     re-reading X from L2);
//   * stages: the depth of the shared-memory ring, from what one stage occupies.
//
// Warp roles (192 threads, persistent, one CTA per SM): warp 0 = TMA producer, warp 1 =
// TMEM allocator + MMA issuer, warps 2..5 = epilogue (tcgen05.ld -> convert -> global).
// Producer and MMA warps run their loops with all 32 lanes converged and let one
// elected lane issue each TMA / tcgen05 instruction.  Full/empty mbarriers guard the
// ring; two TMEM accumulators let the epilogue of tile i overlap the main loop of tile
// i+1.  W layout NK ([N,K]) feeds the MMA
// as a K-major operand with 128-byte swizzle, layout KN ([K,N]) as an N-major operand
// with 64-byte swizzle.  Every mbarrier wait is bounded: a wait that runs out latches
// the device error word, raises a CTA-wide abort flag, drains outstanding copies and
// MMAs (bounded), frees tensor memory and returns.
#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace bi {
namespace {

constexpr int BM = 128;                     // instruction M: token rows
constexpr int BN = 32;                      // instruction N: output columns
constexpr int BK = 64;                      // K-block: one 128-byte swizzle row of bf16
constexpr int UK = 16;                      // K of one kind::f16 instruction
constexpr int MAX_NSUB = 8;
constexpr int MAX_STAGES = 48;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int B_SUB_BYTES = BN * BK * 2;    // 4 KiB: one instruction tile's W block
constexpr int A_MMA_BYTES = BM * BK * 2;    // 16 KiB: what one MMA reads from the X block
constexpr int SMEM_BYTES = 220 * 1024;      // dynamic shared memory per CTA
constexpr int CTRL_BYTES = 1024;            // barriers and flags at the end
constexpr int RING_BYTES = SMEM_BYTES - 1024 /* alignment slack */ - CTRL_BYTES;

static_assert((2 * MAX_STAGES + 5) * 8 + 16 <= CTRL_BYTES, "control block too small");

struct GemmArgs {
    void* y;
    int64_t ldy;
    int M, N, K;
    int a_rows;          // X rows staged per K-block (multiple of 8, <= 128)
    int nsub;            // instruction tiles per CTA tile along N
    int stages;          // ring depth
    int w_stream_once;   // one M-tile: W is read exactly once (L2 evict-first hint)
};

template <bool KN, bool F32OUT>
__global__ void __launch_bounds__(THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            const GemmArgs args, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int S = args.stages;
    const int nsub = args.nsub;
    const int a_bytes = args.a_rows * (BK * 2);
    const int b_bytes = nsub * B_SUB_BYTES;
    const uint32_t stage_tx = uint32_t(a_bytes + b_bytes);
    uint8_t* sA = smem;                         // S x a_bytes
    uint8_t* sB = smem + S * a_bytes;           // S x b_bytes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
    uint64_t* empty = full + MAX_STAGES;
    uint64_t* tfull = empty + MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N, K = args.K;
    const int tile_n = nsub * BN;
    const int m_tiles = (M + BM - 1) / BM;
    const int n_tiles = (N + tile_n - 1) / tile_n;
    const int num_tiles = m_tiles * n_tiles;
    const int nkb = (K + BK - 1) / BK;
    const uint32_t tmem_cols = uint32_t(2 * tile_n);  // two accumulators, power of two

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], EPI_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        latch_error(err, kErrTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer
        // The whole warp runs the loop; one elected lane issues.
        uint32_t stage = 0, phase = 0, issued = 0;
        const uint64_t w_policy = l2_policy_evict_first();
        bool ok = true;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
            const int mt = t / n_tiles, nt = t % n_tiles;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    uint64_t* bar = &full[stage];
                    mbar_arrive_expect_tx(bar, stage_tx);
                    tma_load_2d(sA + stage * a_bytes, &tmap_x, bar, kb * BK, mt * BM);
                    uint8_t* bdst = sB + stage * b_bytes;
                    if (KN) {
                        // one N-major box of 32 columns x 64 k-rows per instruction tile
                        for (int j = 0; j < nsub; ++j) {
                            const int c0 = nt * tile_n + j * BN;
                            if (args.w_stream_once)
                                tma_load_2d_hint(bdst + j * B_SUB_BYTES, &tmap_w, bar, c0, kb * BK,
                                                 w_policy);
                            else
                                tma_load_2d(bdst + j * B_SUB_BYTES, &tmap_w, bar, c0, kb * BK);
                        }
                    } else {
                        // one K-major box of 64 k x (nsub*32) rows covers every instruction tile
                        if (args.w_stream_once)
                            tma_load_2d_hint(bdst, &tmap_w, bar, kb * BK, nt * tile_n, w_policy);
                        else
                            tma_load_2d(bdst, &tmap_w, bar, kb * BK, nt * tile_n);
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == uint32_t(S)) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            if (lane == 0 && !*abort_flag) fail();
            // copies already issued land before the CTA's shared memory is released
            const uint32_t n = issued < uint32_t(S) ? issued : uint32_t(S);
            for (uint32_t i = 1; i <= n; ++i) {
                const uint32_t g = issued - i;
                mbar_wait(&full[g % S], (g / S) & 1u, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop; one elected lane issues the MMAs and commits.
        constexpr uint32_t idesc = umma_idesc_bf16(BM, BN, 0, KN ? 1 : 0);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int local = 0;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + uint32_t(acc * tile_n);
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait_warp(&full[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_addr = smem_addr(sA + stage * a_bytes);
                const uint32_t b_addr = smem_addr(sB + stage * b_bytes);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k) {
                        // X: K-major, 128-byte swizzle, 8-row groups 1024 B apart, +32 B per k16
                        const uint64_t a_desc = umma_smem_desc(a_addr + k * UK * 2, 16, 1024, 2);
                        for (int j = 0; j < nsub; ++j) {
                            uint64_t b_desc;
                            if (KN) {
                                // W: N-major, 64-byte swizzle; k-rows of 64 B, 8 k-rows per
                                // 512-byte atom; a k16 step skips 16 k-rows (1024 B)
                                b_desc = umma_smem_desc(b_addr + j * B_SUB_BYTES + k * UK * 64,
                                                        BK * 64, 512, 4);
                            } else {
                                b_desc = umma_smem_desc(b_addr + j * B_SUB_BYTES + k * UK * 2, 16,
                                                        1024, 2);
                            }
                            tc_mma_bf16(d_tmem + uint32_t(j * BN), a_desc, b_desc, idesc,
                                        (kb | k) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(&empty[stage]);  // frees the stage once these MMAs finish
                }
                __syncwarp();
                if (++stage == uint32_t(S)) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one()) tc_commit(&tfull[acc]);  // accumulator ready for the epilogue
            __syncwarp();
        }
        if (!ok && lane == 0 && !*abort_flag) fail();
        // every MMA this warp issued completes before tensor memory is released
        if (elect_one()) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, nullptr, 100000000ull);
    } else {
        // ------------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const int row_in_tile = quad * 32 + lane;
        int local = 0;
        void* const y = args.y;
        const int64_t ldy = args.ldy;
        const bool vec_ok = F32OUT ? ((ldy % 4) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0)
                                   : ((ldy % 8) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag)) {
                if (!*abort_flag) fail();
                break;
            }
            tc_fence_after_sync();
            const int mt = t / n_tiles, nt = t % n_tiles;
            const int64_t gm = int64_t(mt) * BM + row_in_tile;
            for (int c = 0; c < tile_n; c += 32) {
                uint32_t r[32];
                tmem_load_32x32b_x32(
                    tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * tile_n + c), r);
                tmem_load_wait();
                const int64_t gn0 = int64_t(nt) * tile_n + c;
                if (gm < M && gn0 < N) {
                    if (F32OUT) {
                        float* yr = static_cast<float*>(y) + gm * ldy + gn0;
                        if (vec_ok && gn0 + 32 <= N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4*>(yr + i) =
                                    make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                                __uint_as_float(r[i + 2]),
                                                __uint_as_float(r[i + 3]));
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (gn0 + i < N) yr[i] = __uint_as_float(r[i]);
                        }
                    } else {
                        __nv_bfloat16* yr = static_cast<__nv_bfloat16*>(y) + gm * ldy + gn0;
                        if (vec_ok && gn0 + 32 <= N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                                v.y = pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                                v.z = pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                                v.w = pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                                *reinterpret_cast<uint4*>(yr + i) = v;
                            }
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (gn0 + i < N) yr[i] = __float2bfloat16_rn(__uint_as_float(r[i]));
                        }
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

template <bool KN, bool F32OUT>
cudaError_t launch_t(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                     const GemmArgs& a, int grid, cudaStream_t s) {
    auto kern = gemm_kernel<KN, F32OUT>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    kern<<<grid, THREADS, SMEM_BYTES, s>>>(mx, mw, a, dev.err_word);
    return cudaGetLastError();
}

}  // namespace

int gemm_tile_n() { return BN; }

GemmSchedule gemm_schedule(int64_t M, int64_t N, int num_sms) {
    GemmSchedule g;
    const int64_t m_tiles = (M + BM - 1) / BM;
    g.a_rows = m_tiles == 1 ? int((M + 7) / 8 * 8) : BM;
    // widest CTA tile that still gives every SM a tile (X is then re-read from L2 the
    // fewest times); a single instruction tile per CTA when even that is too few
    g.nsub = 1;
    for (int ns = MAX_NSUB; ns >= 2; ns >>= 1) {
        if (m_tiles * ((N + int64_t(ns) * BN - 1) / (int64_t(ns) * BN)) >= num_sms) {
            g.nsub = ns;
            break;
        }
    }
    const int stage_bytes = g.a_rows * BK * 2 + g.nsub * B_SUB_BYTES;
    g.stages = RING_BYTES / stage_bytes;
    if (g.stages > MAX_STAGES) g.stages = MAX_STAGES;
    g.tiles = m_tiles * ((N + int64_t(g.nsub) * BN - 1) / (int64_t(g.nsub) * BN));
    return g;
}

cudaError_t launch_gemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* w,
                        int64_t ldw, bool w_kn, void* y, int64_t ldy, bool y_f32, int64_t M,
                        int64_t N, int64_t K, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0) {
        // an empty reduction: every output is +0 (all-zero bits in bf16 and fp32)
        const size_t es = y_f32 ? 4 : 2;
        return cudaMemset2DAsync(y, size_t(ldy) * es, 0, size_t(N) * es, size_t(M), stream);
    }
    const GemmSchedule g = gemm_schedule(M, N, dev.num_sms);
    // the MMA of the last stage reads A_MMA_BYTES from its X block: keep that in the ring
    const int a_bytes = g.a_rows * BK * 2;
    if ((g.stages - 1) * a_bytes + A_MMA_BYTES > g.stages * (a_bytes + g.nsub * B_SUB_BYTES) ||
        g.stages < 2)
        return cudaErrorNotSupported;
    CUtensorMap mx, mw;
    if (!tmap_2d_bf16(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK, uint32_t(g.a_rows), 128))
        return cudaErrorNotSupported;
    bool ok;
    if (w_kn)
        ok = tmap_2d_bf16(&mw, w, uint64_t(N), uint64_t(K), uint64_t(ldw), BN, BK, 64);
    else
        ok = tmap_2d_bf16(&mw, w, uint64_t(K), uint64_t(N), uint64_t(ldw), BK,
                          uint32_t(g.nsub * BN), 128);
    if (!ok) return cudaErrorNotSupported;
    GemmArgs a;
    a.y = y;
    a.ldy = ldy;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.a_rows = g.a_rows;
    a.nsub = g.nsub;
    a.stages = g.stages;
    a.w_stream_once = (M + BM - 1) / BM == 1 ? 1 : 0;
    const int grid = int(g.tiles < dev.num_sms ? g.tiles : dev.num_sms);
    if (w_kn)
        return y_f32 ? launch_t<true, true>(dev, mx, mw, a, grid, stream)
                     : launch_t<true, false>(dev, mx, mw, a, grid, stream);
    return y_f32 ? launch_t<false, true>(dev, mx, mw, a, grid, stream)
                 : launch_t<false, false>(dev, mx, mw, a, grid, stream);
}

}  // namespace bi
