// attention.cu -- batch-invariant decode / speculative-verify attention over a bf16 paged
// KV cache: KV append, split-KV partial attention with a FIXED chunk length, and a
// fixed-order log-sum-exp merge.
//
// Sources: "Fix/speculative shape invariance" (ml-explore/mlx PR 4279), Problem (two-pass
// SDPA derives its split count from the query length, changing the softmax tree between
// single-query decoding and multi-query verification) and Changes (a query must reduce
// identically alone or inside a short causal block); book chapter "Batch-invariant
// kernels: why temperature-0 decoding is still nondeterministic", Case 6 strategy table,
// Attention row (update the KV cache before the kernel; fixed split SIZE, varying number
// of splits) and the requirement that token 1000 reduces identically with 0 or 999
// tokens already cached.
//
// Reduction tree of one (query, head) -- a function of the query's position only:
//   * keys are cut into chunks of CHUNK = 512 counted from key 0; the query uses chunks
//     0 .. pos/CHUNK (keys after pos are masked to -inf, so p = +0 exactly);
//   * inside a chunk, 64-key pages 0,2,4,6 are folded by one warp and pages 1,3,5,7 by
//     another, each with an online softmax (running max, exp2 rescale), scores and P.V
//     on the tensor cores (mma.m16n8k16, bf16 in, fp32 accumulate) in a fixed order;
//     the two warp states are then combined, even-page warp first;
//   * chunk partials (m, l, o) are merged by the merge kernel: eight contiguous chunk
//     ranges, each folded in ascending order, then combined in ascending range order --
//     a tree fixed by the number of chunks, i.e. by the query's position.
// A query's row position inside the MMA tile, the number of other queries, sequences,
// or keys beyond pos change none of these steps.
//
// Data movement: one persistent CTA per SM; a producer warp streams K and V pages with
// TMA (2D tensor maps over the cache viewed as [pages*Hkv*PAGE, D], 128-byte swizzle)
// into a 5-deep shared-memory ring; four consumer warps (2 M-tiles x 2 page parities)
// walk every stage in order and compute on the pages of their parity.  Work items (sequence, KV head, chunk) are enumerated on the device
// from seq_lens, so mixed-length batches launch no idle CTAs.
#include "common.cuh"
#include "launch.h"
#include "tmap.h"
#include "bi.h"

namespace bi {
namespace {

constexpr int PAGE = 64;
constexpr int CHUNK = 512;
constexpr int PAGES_PER_CHUNK = CHUNK / PAGE;
constexpr int MAXR = 32;       // query rows per (sequence, KV head): q_len * group size
constexpr int NCONS = 4;       // consumer warps
constexpr int THREADS = (NCONS + 1) * 32;
constexpr int NST = 5;         // page stages in the ring
constexpr int MAX_BATCH = BI_ATTN_MAX_BATCH;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

static_assert(CHUNK % PAGE == 0, "chunk must hold whole pages");

template <int D>
struct Cfg {
    static constexpr int BOXES = D / 64;                // 64-element (128 B) column boxes
    static constexpr int BOX_BYTES = PAGE * 128;        // one box of a page: 64 rows x 128 B
    static constexpr int PAGE_BYTES = BOXES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;  // K page + V page
    static constexpr int QBOX_BYTES = MAXR * 128;
    static constexpr int Q_BYTES = BOXES * QBOX_BYTES;
    static constexpr int NDN = D / 8;                   // 8-wide column tiles of O
    static constexpr int COMB_O_BYTES = 2 * NDN * 32 * 16;
    static constexpr int COMB_ML_BYTES = 2 * 32 * 16;
    static constexpr size_t SMEM = 1024 + size_t(NST) * STAGE_BYTES + Q_BYTES + COMB_O_BYTES +
                                   COMB_ML_BYTES + 2 * NST * 8 + NST * 4 + (MAX_BATCH + 1) * 4 +
                                   64;
};

// byte offset of (row, 16-byte chunk) in a 128-byte-swizzled box (the TMA SWIZZLE_128B
// pattern: chunk index XOR row mod 8)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return uint32_t(row) * 128u + (uint32_t((chunk ^ (row & 7)) & 7) << 4);
}

__device__ __forceinline__ void named_barrier_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCONS * 32) : "memory");
}

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

// ------------------------------------------------------------------- partial kernel

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_partial_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
                    int max_pages, int num_pages, const int32_t* __restrict__ seq_lens,
                    const int32_t* __restrict__ cu_q, int B, int total_q, int max_q,
                    int max_seq_len, int Hq, int Hkv, float scale_log2,
                    float* __restrict__ ws_o, float* __restrict__ ws_ml, int maxC,
                    unsigned int* err) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sStage = smem;
    uint8_t* sQ = sStage + NST * C::STAGE_BYTES;
    float4* comb_o = reinterpret_cast<float4*>(sQ + C::Q_BYTES);
    float4* comb_ml = reinterpret_cast<float4*>(sQ + C::Q_BYTES + C::COMB_O_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(sQ + C::Q_BYTES + C::COMB_O_BYTES +
                                                 C::COMB_ML_BYTES);
    uint64_t* empty = full + NST;
    int* stage_valid = reinterpret_cast<int*>(empty + NST);
    int* prefix = stage_valid + NST;  // [B+1]
    volatile int* abort_flag = prefix + MAX_BATCH + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv;

    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            // every consumer warp releases every stage (also pages of the other parity),
            // so no warp can run a full ring cycle ahead and alias an mbarrier phase
            mbar_init(&empty[s], NCONS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // work items per sequence: chunks x KV heads (0 for a malformed sequence)
    for (int b = tid; b < B; b += THREADS) {
        const SeqInfo s = seq_info(seq_lens, cu_q, b);
        const bool ok = seq_ok(s, max_q, max_seq_len, total_q);
        if (!ok) latch_error(err, kErrDeviceArg);
        prefix[b + 1] = ok ? ((s.L + CHUNK - 1) / CHUNK) * Hkv : 0;
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of prefix[1..B], 32 at a time
        int carry = 0;
        for (int base = 0; base < B; base += 32) {
            const int i = base + lane;
            int v = i < B ? prefix[i + 1] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += u;
            }
            if (i < B) prefix[i + 1] = v + carry;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) prefix[0] = 0;
    }
    __syncthreads();
    const int total = prefix[B];

    auto decode = [&](int w, int& b, int& c, int& h) {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= w) lo = mid; else hi = mid;
        }
        b = lo;
        const int r = w - prefix[b];
        c = r / Hkv;
        h = r - c * Hkv;
    };

    if (warp == NCONS) {
        // ------------------------------------------------------------------ producer
        // The whole warp runs the loop (converged, warp-uniform state); one elected lane
        // reads the page index and issues the copies.
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        uint32_t g = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
            int b, c, h;
            decode(w, b, c, h);
            const SeqInfo si = seq_info(seq_lens, cu_q, b);
            const int npages = min(PAGES_PER_CHUNK, (si.L - c * CHUNK + PAGE - 1) / PAGE);
            for (int i = 0; i < npages; ++i, ++g) {
                const int s = int(g % NST);
                const uint32_t ph = (g / NST) & 1u;
                if (!mbar_wait_warp(&empty[s], ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const int pidx = c * PAGES_PER_CHUNK + i;
                    const int phys =
                        pidx < max_pages ? block_table[int64_t(b) * max_pages + pidx] : -1;
                    const bool valid = phys >= 0 && phys < num_pages;
                    stage_valid[s] = valid ? 1 : 0;
                    if (valid) {
                        uint8_t* st = sStage + s * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                        const int row = (phys * Hkv + h) * PAGE;
#pragma unroll
                        for (int bx = 0; bx < C::BOXES; ++bx) {
                            tma_load_2d(st + bx * C::BOX_BYTES, &tmap_k, &full[s], bx * 64, row);
                            tma_load_2d(st + C::PAGE_BYTES + bx * C::BOX_BYTES, &tmap_v, &full[s],
                                        bx * 64, row);
                        }
                    } else {
                        latch_error(err, kErrDeviceArg);
                        mbar_arrive(&full[s]);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                latch_error(err, kErrTimeout);
            }
            // copies already issued land before the CTA exits (bounded)
            for (int k = 1; k <= NST && k <= int(g); ++k) {
                const uint32_t gg = g - k;
                mbar_wait(&full[gg % NST], (gg / NST) & 1u, nullptr, 100000000ull);
            }
        }
        return;  // the producer takes no part in the consumers' named barriers
    }

    // ---------------------------------------------------------------------- consumers
    const int mt = warp & 1;   // M-tile: query rows 16*mt .. 16*mt+15
    const int par = warp >> 1; // page parity folded by this warp
    const int quad_row = lane >> 2;
    const int quad_col = (lane & 3) * 2;
    const uint32_t sQa = smem_addr(sQ);
    uint32_t g = 0;
    bool alive = true;

    for (int w = blockIdx.x; w < total; w += gridDim.x) {
        int b, c, h;
        decode(w, b, c, h);
        const SeqInfo si = seq_info(seq_lens, cu_q, b);
        const int L = si.L, qb = si.qb;
        const int npages = min(PAGES_PER_CHUNK, (L - c * CHUNK + PAGE - 1) / PAGE);
        const int R = qb * G;
        const bool active = alive && (mt * 16 < R);

        // Q tile of (sequence b, KV head h): row r = j*G + gg, zero past R
        named_barrier_consumers();
        for (int idx = tid; idx < MAXR * (D / 8); idx += NCONS * 32) {
            const int r = idx / (D / 8), ch = idx - r * (D / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < R) {
                const int j = r / G, gg = r - j * G;
                const int64_t off = (int64_t(si.t0 + j) * Hq + int64_t(h) * G + gg) * D + ch * 8;
                v = *reinterpret_cast<const uint4*>(q + off);
            }
            *reinterpret_cast<uint4*>(sQ + (ch >> 3) * C::QBOX_BYTES + swz(r, ch & 7)) = v;
        }
        named_barrier_consumers();

        const int rA = mt * 16 + quad_row, rB = rA + 8;
        const int posA = rA < R ? L - qb + rA / G : -1;
        const int posB = rB < R ? L - qb + rB / G : -1;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        float o[C::NDN][4];
#pragma unroll
        for (int dn = 0; dn < C::NDN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

        for (int i = 0; i < npages; ++i) {
            const uint32_t gi = g + i;
            const int s = int(gi % NST);
            if (alive && !mbar_wait_warp(&full[s], (gi / NST) & 1u, abort_flag)) {
                alive = false;
                if (!*abort_flag) {
                    *abort_flag = 1;
                    latch_error(err, kErrTimeout);
                }
            }
            if ((i & 1) == par && active && alive && stage_valid[s]) {
                const int page_base = c * CHUNK + i * PAGE;
                const uint32_t kb = smem_addr(sStage + s * C::STAGE_BYTES);
                const uint32_t vb = kb + C::PAGE_BYTES;
                // ---- S = Q K^T (16 rows x 64 keys), fp32
                float sc[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a[4];
                    {
                        const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                        const int dch = kk * 2 + (lane >> 4);
                        ldmatrix_x4(sQa + (dch >> 3) * C::QBOX_BYTES + swz(r, dch & 7), a[0], a[1],
                                    a[2], a[3]);
                    }
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        const int mi = lane >> 3;
                        const int key = np * 16 + (lane & 7) + (mi >> 1) * 8;
                        const int dch = kk * 2 + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kb + (dch >> 3) * C::BOX_BYTES + swz(key, dch & 7), b0, b1, b2,
                                    b3);
                        mma_bf16_16816(sc[2 * np], a, b0, b1);
                        mma_bf16_16816(sc[2 * np + 1], a, b2, b3);
                    }
                }
                // ---- scale (log2 domain), causal mask, row max
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = page_base + nt * 8 + quad_col + (e & 1);
                        const int pos = e < 2 ? posA : posB;
                        const float v = key <= pos ? sc[nt][e] * scale_log2 : -INFINITY;
                        sc[nt][e] = v;
                        mx[e >> 1] = fmaxf(mx[e >> 1], v);
                    }
                }
                float alpha[2], m_use[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
                    mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
                    const float m_new = fmaxf(m_run[hh], mx[hh]);
                    m_use[hh] = m_new == -INFINITY ? 0.f : m_new;
                    alpha[hh] = exp2f(m_run[hh] - m_use[hh]);
                    m_run[hh] = m_new;
                }
                // ---- p = exp2(s - m), row sums in a fixed order, P packed to bf16
                float ps[2] = {0.f, 0.f};
                uint32_t pa[8][2];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const float p0 = exp2f(sc[nt][0] - m_use[0]);
                    const float p1 = exp2f(sc[nt][1] - m_use[0]);
                    const float p2 = exp2f(sc[nt][2] - m_use[1]);
                    const float p3 = exp2f(sc[nt][3] - m_use[1]);
                    ps[0] = ps[0] + p0;
                    ps[0] = ps[0] + p1;
                    ps[1] = ps[1] + p2;
                    ps[1] = ps[1] + p3;
                    pa[nt][0] = pack_bf16x2(p0, p1);
                    pa[nt][1] = pack_bf16x2(p2, p3);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    ps[hh] += __shfl_xor_sync(0xffffffffu, ps[hh], 1);
                    ps[hh] += __shfl_xor_sync(0xffffffffu, ps[hh], 2);
                    l_run[hh] = l_run[hh] * alpha[hh] + ps[hh];
                }
#pragma unroll
                for (int dn = 0; dn < C::NDN; ++dn) {
                    o[dn][0] *= alpha[0];
                    o[dn][1] *= alpha[0];
                    o[dn][2] *= alpha[1];
                    o[dn][3] *= alpha[1];
                }
                // ---- O += P V (keys as K dimension); V rows past the sequence end are
                // zeroed so unwritten cache slots cannot inject NaN/Inf through 0 * v
                const bool tail = page_base + PAGE > L;
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const uint32_t a[4] = {pa[2 * k2][0], pa[2 * k2][1], pa[2 * k2 + 1][0],
                                           pa[2 * k2 + 1][1]};
                    const int klo = page_base + k2 * 16 + quad_col;  // keys of b0 (b1: +8)
#pragma unroll
                    for (int dp = 0; dp < C::NDN / 2; ++dp) {
                        const int mi = lane >> 3;
                        const int key = k2 * 16 + (lane & 7) + (mi & 1) * 8;
                        const int dch = dp * 2 + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(vb + (dch >> 3) * C::BOX_BYTES + swz(key, dch & 7), b0,
                                          b1, b2, b3);
                        if (tail) {
                            const uint32_t m0 = (klo < L ? 0x0000ffffu : 0u) |
                                                (klo + 1 < L ? 0xffff0000u : 0u);
                            const uint32_t m1 = (klo + 8 < L ? 0x0000ffffu : 0u) |
                                                (klo + 9 < L ? 0xffff0000u : 0u);
                            b0 &= m0;
                            b2 &= m0;
                            b1 &= m1;
                            b3 &= m1;
                        }
                        mma_bf16_16816(o[2 * dp], a, b0, b1);
                        mma_bf16_16816(o[2 * dp + 1], a, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        g += npages;

        // ---- combine the two page parities (even pages first) and write the partial
        if (par == 1 && active) {
#pragma unroll
            for (int dn = 0; dn < C::NDN; ++dn)
                comb_o[(mt * C::NDN + dn) * 32 + lane] = make_float4(o[dn][0], o[dn][1], o[dn][2],
                                                                     o[dn][3]);
            comb_ml[mt * 32 + lane] = make_float4(m_run[0], m_run[1], l_run[0], l_run[1]);
        }
        named_barrier_consumers();
        if (par == 0 && active) {
            const float4 mlB = comb_ml[mt * 32 + lane];
            const float mB[2] = {mlB.x, mlB.y}, lB[2] = {mlB.z, mlB.w};
            float wa[2], wb[2], mm[2], ll[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                mm[hh] = fmaxf(m_run[hh], mB[hh]);
                if (mm[hh] == -INFINITY) {
                    wa[hh] = 0.f;
                    wb[hh] = 0.f;
                } else {
                    wa[hh] = exp2f(m_run[hh] - mm[hh]);
                    wb[hh] = exp2f(mB[hh] - mm[hh]);
                }
                ll[hh] = l_run[hh] * wa[hh] + lB[hh] * wb[hh];
            }
            const int rows[2] = {rA, rB};
            const int poss[2] = {posA, posB};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = rows[hh];
                if (r >= R || poss[hh] < c * CHUNK) continue;
                const int j = r / G, gg = r - j * G;
                const int64_t idx = (int64_t(si.t0 + j) * Hq + int64_t(h) * G + gg) * maxC + c;
                float* dst = ws_o + idx * D + quad_col;
#pragma unroll
                for (int dn = 0; dn < C::NDN; ++dn) {
                    const float4 ob = comb_o[(mt * C::NDN + dn) * 32 + lane];
                    const float obv0 = hh == 0 ? ob.x : ob.z;
                    const float obv1 = hh == 0 ? ob.y : ob.w;
                    const float v0 = o[dn][2 * hh] * wa[hh] + obv0 * wb[hh];
                    const float v1 = o[dn][2 * hh + 1] * wa[hh] + obv1 * wb[hh];
                    *reinterpret_cast<float2*>(dst + dn * 8) = make_float2(v0, v1);
                }
                if ((lane & 3) == 0)
                    *reinterpret_cast<float2*>(ws_ml + idx * 2) = make_float2(mm[hh], ll[hh]);
            }
        }
    }
}

// --------------------------------------------------------------------- merge kernel

constexpr int MERGE_WARPS = 8;

// One CTA per (token, query head) merges the chunk partials 0 .. nC-1 (nC = pos/CHUNK+1).
// Warp w folds the contiguous range [w*nC/8, (w+1)*nC/8) in ascending order (max first,
// then the exp2-weighted sums); the eight warp results are combined in ascending warp
// order.  The tree is a function of nC alone, i.e. of the query's position.
template <int D>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
attn_merge_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
                  int total_q, int max_q, int max_seq_len, int Hq,
                  const float* __restrict__ ws_o, const float* __restrict__ ws_ml, int maxC,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    constexpr int PER = D / 32;
    constexpr int UNROLL = 4;
    __shared__ float sM[MERGE_WARPS], sL[MERGE_WARPS];
    __shared__ float sO[MERGE_WARPS][D];
    pdl_wait();
    pdl_trigger();
    const int t = int(blockIdx.x / unsigned(Hq));
    const int hq = int(blockIdx.x - unsigned(t) * unsigned(Hq));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int b;
    if (cu_q) {
        int lo = 0, hi = B;  // largest b with cu_q[b] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_q[mid] <= t) lo = mid; else hi = mid;
        }
        b = lo;
    } else {
        b = t;
    }
    const SeqInfo si = seq_info(seq_lens, cu_q, b);
    if (!seq_ok(si, max_q, max_seq_len, total_q) || t < si.t0 || t >= si.t0 + si.qb) return;
    const int pos = si.L - si.qb + (t - si.t0);
    const int nC = pos / CHUNK + 1;
    const int64_t base = (int64_t(t) * Hq + hq) * maxC;
    const int c0 = warp * nC / MERGE_WARPS, c1 = (warp + 1) * nC / MERGE_WARPS;

    // range max: lanes stride over chunks, then a butterfly (max is exact)
    float Mw = -INFINITY;
    for (int c = c0 + lane; c < c1; c += 32) Mw = fmaxf(Mw, ws_ml[(base + c) * 2]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, off));

    float Lw = 0.f;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int c = c0; c < c1; c += UNROLL) {
        float v[UNROLL][PER];
        float2 ml[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {  // issue the loads of UNROLL chunks first
            if (c + u < c1) {
                ml[u] = *reinterpret_cast<const float2*>(ws_ml + (base + c + u) * 2);
                const float* src = ws_o + (base + c + u) * D + lane * PER;
                if (PER == 4) {
                    const float4 f = *reinterpret_cast<const float4*>(src);
                    v[u][0] = f.x; v[u][1 % PER] = f.y; v[u][2 % PER] = f.z; v[u][3 % PER] = f.w;
                } else {
                    const float2 f = *reinterpret_cast<const float2*>(src);
                    v[u][0] = f.x; v[u][1 % PER] = f.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {  // then fold them in ascending chunk order
            if (c + u < c1) {
                const float wgt = exp2f(ml[u].x - Mw);
                Lw = Lw + wgt * ml[u].y;
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] = acc[i] + wgt * v[u][i];
            }
        }
    }
    if (lane == 0) {
        sM[warp] = Mw;
        sL[warp] = Lw;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) sO[warp][lane * PER + i] = acc[i];
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) M = fmaxf(M, sM[w]);
    float L = 0.f;
    float o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = 0.f;
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) {
        const float wgt = exp2f(sM[w] - M);  // an empty range has sM = -inf: weight 0
        L = L + wgt * sL[w];
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = o[i] + wgt * sO[w][lane * PER + i];
    }
    __nv_bfloat16* dst = out + (int64_t(t) * Hq + hq) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[i] = __float2bfloat16_rn(o[i] / L);
    if (lse && lane == 0) lse[int64_t(t) * Hq + hq] = (M + log2f(L)) * kLn2;
}

// ------------------------------------------------------------------ KV-append kernel

__global__ void __launch_bounds__(256)
kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_pages,
                 const int32_t* __restrict__ block_table, int max_pages,
                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
                 int total_q, int Hkv, int D, unsigned int* err) {
    // one thread per 16-byte piece of one token's K (and V) row of one KV head
    pdl_wait();
    pdl_trigger();
    const int per_tok = Hkv * (D / 8);
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= int64_t(total_q) * per_tok) return;
    const int t = int(idx / per_tok);
    const int rem = int(idx - int64_t(t) * per_tok);
    const int h = rem / (D / 8), ch = rem - h * (D / 8);
    int lo = 0, hi = B;  // sequence of token t: largest b with cu_q[b] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu_q[mid] <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int L = seq_lens[b];
    const int t0 = cu_q[b];
    const int qb = cu_q[b + 1] - t0;
    if (t < t0 || t >= t0 + qb) return;  // token of no sequence (cu_q[0] > 0)
    if (qb > L || L > max_pages * PAGE || t0 + qb > total_q) {
        latch_error(err, kErrDeviceArg);
        return;
    }
    const int pos = L - qb + (t - t0);
    const int phys = block_table[int64_t(b) * max_pages + pos / PAGE];
    if (phys < 0 || phys >= num_pages) {
        latch_error(err, kErrDeviceArg);
        return;
    }
    const int64_t dst = ((int64_t(phys) * Hkv + h) * PAGE + pos % PAGE) * (D / 8) + ch;
    const int64_t src = (int64_t(t) * Hkv + h) * (D / 8) + ch;
    k_cache[dst] = k_new[src];
    v_cache[dst] = v_new[src];
}

template <int D>
cudaError_t launch_attention_t(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                               float scale, void* out, float* lse, void* workspace,
                               cudaStream_t stream) {
    using Cf = Cfg<D>;
    const uint64_t rows = uint64_t(a.num_pages) * uint64_t(a.hkv) * PAGE;
    CUtensorMap tk, tv;
    if (!tmap_2d_bf16(&tk, a.k_cache, D, rows, D, 64, PAGE, 128) ||
        !tmap_2d_bf16(&tv, a.v_cache, D, rows, D, 64, PAGE, 128))
        return cudaErrorNotSupported;
    auto kern = attn_partial_kernel<D>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(Cf::SMEM));
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    const int maxC = int((a.max_seq_len + CHUNK - 1) / CHUNK);
    const int64_t items_bound = a.batch * int64_t(maxC) * a.hkv;
    if (items_bound > 0x7fffffffLL) return cudaErrorNotSupported;
    const int grid = int(items_bound < dev.num_sms ? items_bound : dev.num_sms);
    float* ws_o = static_cast<float*>(workspace);
    float* ws_ml = ws_o + a.total_q * a.hq * int64_t(maxC) * D;
    const float scale_log2 = scale * kLog2e;
    cudaError_t e = launch_pdl(
        kern, dim3(grid), dim3(THREADS), Cf::SMEM, stream, tk, tv,
        static_cast<const __nv_bfloat16*>(q), a.block_table, int(a.max_pages), int(a.num_pages),
        a.seq_lens, a.cu_q, int(a.batch), int(a.total_q), int(a.max_q), int(a.max_seq_len),
        int(a.hq), int(a.hkv), scale_log2, ws_o, ws_ml, maxC, dev.err_word);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_merge_kernel<D>, dim3(unsigned(a.total_q * a.hq)),
                      dim3(MERGE_WARPS * 32), 0, stream, a.seq_lens, a.cu_q, int(a.batch),
                      int(a.total_q), int(a.max_q), int(a.max_seq_len), int(a.hq),
                      static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml), maxC,
                      static_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace

size_t attn_workspace_bytes(int64_t total_q, int64_t hq, int64_t head_dim, int64_t max_seq_len) {
    const int64_t chunks = (max_seq_len + CHUNK - 1) / CHUNK;
    return size_t(total_q) * size_t(hq) * size_t(chunks) * size_t(head_dim + 2) * sizeof(float);
}

cudaError_t launch_kv_append(const DeviceInfo& dev, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, const PagedArgs& a,
                             cudaStream_t stream) {
    const int64_t n = a.total_q * a.hkv * (a.head_dim / 8);
    return launch_pdl(kv_append_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, stream,
                      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                      int(a.num_pages), a.block_table, int(a.max_pages), a.seq_lens, a.cu_q,
                      int(a.batch), int(a.total_q), int(a.hkv), int(a.head_dim), dev.err_word);
}

cudaError_t launch_attention(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                             float scale, void* out, float* lse, void* workspace,
                             cudaStream_t stream) {
    if (a.head_dim == 64) return launch_attention_t<64>(dev, q, a, scale, out, lse, workspace, stream);
    return launch_attention_t<128>(dev, q, a, scale, out, lse, workspace, stream);
}

}  // namespace bi
