// gemm.cu -- batch-invariant bf16 GEMM on the 5th-generation tensor cores (tcgen05).
//
// Sources: book chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Case 3 (a K tile picked from the batch size changes row 0) and the
// Case 6 strategy table, Matmul row (one compiled configuration for all shapes, no
// Split-K, no switch to a narrower instruction for small M); "Fix/speculative shape
// invariance" (ml-explore/mlx PR 4279), Problem (GEMV vs gemv_wide vs GEMM chosen by the
// row count is the defect) and the review thread (both B orientations must be covered).
//
// Design (one configuration for every M):
//   * Output tile 128 x BN.  Each tile is accumulated in tensor memory (fp32) by
//     tcgen05.mma.cta_group::1.kind::f16 instructions of shape 128 x BN x 16, issued for
//     K-blocks of 64 in ascending order and, inside a block, for k = 0,16,32,48 in order.
//     Row m of Y is always lane m%128 of M-tile m/128; rows past M are zero-filled by
//     TMA and never stored.  Nothing about the instruction stream of a tile depends on M.
//   * Warp roles (192 threads, persistent, one CTA per SM): warp 0 = TMA producer,
//     warp 1 = TMEM allocator + single-thread MMA issuer, warps 2..5 = epilogue
//     (tcgen05.ld -> fp32 -> bf16 RNE -> global).  A STAGES-deep shared-memory ring
//     of (X block, W block) pairs is guarded by full/empty mbarriers; two TMEM
//     accumulators let the epilogue of tile i overlap the main loop of tile i+1.
//   * W layout NK ([N,K], K contiguous) feeds the MMA as a K-major operand; layout KN
//     ([K,N], N contiguous) as an N-major operand.  Both use the 128-byte (or, for a
//     32-wide tile, 64-byte) swizzle that TMA writes and the UMMA descriptor reads.
//   * Every mbarrier wait is bounded; a wait that runs out latches the device error
//     word, raises a CTA-wide abort flag, drains outstanding copies / MMAs (bounded),
//     frees its tensor memory and returns.
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "launch.h"

#ifndef BI_GEMM_BN
#define BI_GEMM_BN 32
#endif

namespace bi {
namespace {

constexpr int BM = 128;
constexpr int BN = BI_GEMM_BN;
constexpr int BK = 64;        // one 128-byte swizzle row of bf16
constexpr int UK = 16;        // K of one kind::f16 instruction
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BUDGET = 220 * 1024;
constexpr int STAGES = (SMEM_BUDGET - 1024) / STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;

static_assert(BN == 32 || BN == 64, "tile N must be 32 or 64 (one swizzle atom per k-row)");
static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM alloc size");
static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte swizzle alignment");
static_assert(STAGES >= 4, "pipeline too shallow");

// Swizzle of the N-major W tile in shared memory: BN bf16 = BN*2 bytes per k-row.
constexpr int KN_SWIZZLE_BYTES = BN * 2 >= 128 ? 128 : BN * 2;
constexpr uint32_t KN_LAYOUT = KN_SWIZZLE_BYTES == 128 ? 2u : (KN_SWIZZLE_BYTES == 64 ? 4u : 6u);

constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + size_t(STAGES) * STAGE_BYTES +
           (2 * STAGES + 5) * sizeof(uint64_t) + 16;
}

struct Pipe {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

template <bool KN, bool F32OUT>
__global__ void __launch_bounds__(THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            void* __restrict__ y, int64_t ldy, int M, int N, int K, int w_stream_once,
            unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m_tiles = (M + BM - 1) / BM;
    const int n_tiles = (N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int nkb = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
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
        tmem_alloc(tmem_slot, TMEM_COLS);
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
        if (lane == 0) {
            Pipe p;
            uint32_t issued_phase[STAGES];
            bool issued[STAGES];
            for (int s = 0; s < STAGES; ++s) issued[s] = false;
            const uint64_t w_policy = l2_policy_evict_first();
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                const int mt = t / n_tiles, nt = t % n_tiles;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[p.stage], p.phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint64_t* bar = &full[p.stage];
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    tma_load_2d(sA + p.stage * A_BYTES, &tmap_x, bar, kb * BK, mt * BM);
                    const int wc0 = KN ? nt * BN : kb * BK;
                    const int wc1 = KN ? kb * BK : nt * BN;
                    // W is read exactly once when there is a single M-tile: keep it from
                    // displacing X in L2.  (A cache hint; it never changes any value.)
                    if (w_stream_once)
                        tma_load_2d_hint(sB + p.stage * B_BYTES, &tmap_w, bar, wc0, wc1, w_policy);
                    else
                        tma_load_2d(sB + p.stage * B_BYTES, &tmap_w, bar, wc0, wc1);
                    issued[p.stage] = true;
                    issued_phase[p.stage] = p.phase;
                    p.advance();
                }
            }
            if (!ok) {
                if (!*abort_flag) fail();
                // let copies already in flight land before the CTA's smem is released
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s]) mbar_wait(&full[s], issued_phase[s], nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(BM, BN, 0, KN ? 1 : 0);
            Pipe p;
            bool ok = true;
            int local = 0;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[p.stage], p.phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_addr(sA + p.stage * A_BYTES);
                    const uint32_t b_addr = smem_addr(sB + p.stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k) {
                        // A: K-major, 128B swizzle, 8-row groups 1024 B apart; +32 B per k16
                        const uint64_t a_desc = umma_smem_desc(a_addr + k * UK * 2, 16, 1024, 2);
                        uint64_t b_desc;
                        if (KN) {
                            // B: N-major; each k-row is BN*2 bytes, 8 k-rows per swizzle atom;
                            // a k16 step skips 16 k-rows.
                            b_desc = umma_smem_desc(b_addr + k * UK * (BN * 2),
                                                    BK * KN_SWIZZLE_BYTES, 8 * KN_SWIZZLE_BYTES,
                                                    KN_LAYOUT);
                        } else {
                            b_desc = umma_smem_desc(b_addr + k * UK * 2, 16, 1024, 2);
                        }
                        tc_mma_bf16(d_tmem, a_desc, b_desc, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[p.stage]);  // frees the stage once these MMAs finish
                    p.advance();
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);  // accumulator ready for the epilogue
            }
            if (!ok && !*abort_flag) fail();
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr, 100000000ull);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const int row_in_tile = quad * 32 + lane;
        int local = 0;
        const bool vec_ok = F32OUT ? ((ldy % 4) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0)
                                   : ((ldy % 8) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
                if (!*abort_flag) fail();
                break;
            }
            tc_fence_after_sync();
            const int mt = t / n_tiles, nt = t % n_tiles;
            const int64_t gm = int64_t(mt) * BM + row_in_tile;
#pragma unroll
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_load_32x32b_x32(tmem_base + (uint32_t(quad * 32) << 16) + acc * BN + c, r);
                tmem_load_wait();
                const int64_t gn0 = int64_t(nt) * BN + c;
                if (gm < M) {
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
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------ TMA descriptor cache

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

struct MapKey {
    uintptr_t ptr;
    uint64_t inner, outer, stride;
    uint32_t box_inner, box_outer, swizzle;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && stride == o.stride &&
               box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        h ^= k.inner + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= k.outer + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= k.stride + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
        h ^= (uint64_t(k.box_inner) << 32 | k.box_outer) + (h << 6) + (h >> 2);
        return size_t(h ^ k.swizzle);
    }
};

std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// 2D bf16 tensor [outer][inner] with a row stride of `stride` elements.
bool get_map_2d(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer, uint64_t stride,
                uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
    const MapKey key{reinterpret_cast<uintptr_t>(ptr), inner, outer, stride, box_inner, box_outer,
                     uint32_t(swizzle_bytes)};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return true;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B;
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return true;
}

template <bool KN, bool F32OUT>
cudaError_t launch_t(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw, void* y,
                     int64_t ldy, int M, int N, int K, cudaStream_t s) {
    auto kern = gemm_kernel<KN, F32OUT>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem_bytes()));
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = tiles < dev.num_sms ? tiles : dev.num_sms;
    const int w_once = (M + BM - 1) / BM == 1 ? 1 : 0;
    kern<<<grid, THREADS, smem_bytes(), s>>>(mx, mw, y, ldy, M, N, K, w_once, dev.err_word);
    return cudaGetLastError();
}

}  // namespace

int gemm_tile_n() { return BN; }

cudaError_t launch_gemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* w,
                        int64_t ldw, bool w_kn, void* y, int64_t ldy, bool y_f32, int64_t M,
                        int64_t N, int64_t K, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0) {
        // an empty reduction: every output is +0 (all-zero bits in bf16 and fp32)
        const size_t es = y_f32 ? 4 : 2;
        return cudaMemset2DAsync(y, size_t(ldy) * es, 0, size_t(N) * es, size_t(M), stream);
    }
    CUtensorMap mx, mw;
    if (!get_map_2d(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK, BM, 128))
        return cudaErrorNotSupported;
    bool ok;
    if (w_kn)
        ok = get_map_2d(&mw, w, uint64_t(N), uint64_t(K), uint64_t(ldw), BN, BK, KN_SWIZZLE_BYTES);
    else
        ok = get_map_2d(&mw, w, uint64_t(K), uint64_t(N), uint64_t(ldw), BK, BN, 128);
    if (!ok) return cudaErrorNotSupported;
    const int m = int(M), n = int(N), k = int(K);
    if (w_kn)
        return y_f32 ? launch_t<true, true>(dev, mx, mw, y, ldy, m, n, k, stream)
                     : launch_t<true, false>(dev, mx, mw, y, ldy, m, n, k, stream);
    return y_f32 ? launch_t<false, true>(dev, mx, mw, y, ldy, m, n, k, stream)
                 : launch_t<false, false>(dev, mx, mw, y, ldy, m, n, k, stream);
}

}  // namespace bi
