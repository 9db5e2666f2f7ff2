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
//   * per 64-key page, the scores S = Q K^T come from tcgen05 MMAs (bf16 in, fp32
//     accumulate in tensor memory; head-dim steps of 16 in ascending order);
//   * the chunk's pages are folded in ascending order with an online softmax against a
//     reference max m that is raised only when a page's row max exceeds it by more than
//     2^8 (then O and the row sums are rescaled by 2^(m_old - m_new)); P = 2^(S - m)
//     (both powers by the hardware's ex2 approximation, see attn_common.cuh)
//     is rounded to bf16 and O += P V accumulates in tensor memory (tcgen05, the page's
//     keys in 16-key steps, ascending); each of four warps sums its 16-key slice of the
//     row key by key, and the four slice sums are added in ascending slice order;
//   * chunk partials (m, l, o) are merged by the merge kernel: eight contiguous chunk
//     ranges, each folded in ascending order, then combined in ascending range order --
//     a tree fixed by the number of chunks, i.e. by the query's position.
// A query's row inside the MMA tile, the number of other queries, sequences, or keys
// beyond pos change none of these steps.
//
// Data movement: one persistent CTA of seven warps per SM.  Warp 5 streams K and V pages
// with TMA (2D tensor maps over the cache viewed as [pages*Hkv*PAGE, D], 128-byte
// swizzle) into a shared-memory ring; warp 6 issues the MMAs (S into a double-buffered
// tensor-memory tile, then P V into a per-item fp32 O accumulator, double-buffered);
// warps 0..3 run the softmax, each on a 16-key slice of every page (the <= 32 query rows
// are repeated in each of the four tensor-memory lane quarters); warp 4 reads each
// finished O out and writes the chunk partial while the next item runs.  Work items (sequence, KV head, chunk) are
// enumerated on the device from seq_lens, so mixed-length batches launch no idle CTAs.
#include "attn_common.cuh"

namespace bi {
namespace {

constexpr int MIN_CHUNK_LOG2 = 6, MAX_CHUNK_LOG2 = 11;  // non-invariant calls: 64 .. 2048
constexpr int PV_LAG = 2;      // P V of page g is issued after S of page g+2
constexpr int MAXR = 32;       // query rows per (sequence, KV head): q_len * group size
constexpr int NSM = 4;         // softmax warps 0..3, one per tensor-memory lane quarter
constexpr int KSL = PAGE / NSM;  // keys of a page per softmax warp
constexpr int EPILOGUE = NSM;  // reads O (lanes 0..31: a warp whose index is 0 mod 4)
constexpr int PRODUCER = NSM + 1, MMA_WARP = NSM + 2;
constexpr int THREADS = (NSM + 3) * 32;
constexpr int MMA_M = 128;     // instruction rows: Q rows repeated once per lane quarter
constexpr int TMEM_COLS = 512;
constexpr int MAX_BATCH = BI_ATTN_MAX_BATCH;

static_assert(CHUNK % PAGE == 0, "chunk must hold whole pages");
static_assert(PAGE == 64 && KSL == 16, "a page is one 64-column S tile, 16 keys per warp");
static_assert(NSM * MAXR == MMA_M, "one copy of the query rows per lane quarter");
static_assert(EPILOGUE % 4 == 0, "the epilogue warp must own tensor-memory lanes 0..31");

template <int D>
struct Cfg {
    static constexpr int NST = D == 64 ? 8 : 5;         // page stages in the ring
    static constexpr int BOXES = D / 64;                // 64-element (128 B) column boxes
    static constexpr int BOX_BYTES = PAGE * 128;        // one box of a page: 64 rows x 128 B
    static constexpr int PAGE_BYTES = BOXES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;  // K page + V page
    static constexpr int QBOX_BYTES = MMA_M * 128;      // 128 rows: the MAXR rows, 4 times
    static constexpr int Q_BYTES = BOXES * QBOX_BYTES;
    // P holds MAXR real rows.  An M = 128 MMA reads 128 rows (16 KB) from its base; rows
    // >= MAXR only feed accumulator rows that are never read, so that read may run on
    // into the ring, which follows and is larger than 16 KB.
    static constexpr int P_BYTES = MAXR * 128;
    static constexpr int RING_OFF = Q_BYTES + 2 * P_BYTES;
    static constexpr int BAR_OFF = RING_OFF + NST * STAGE_BYTES;
    static constexpr int NBARS = 2 * NST + 14 + 2;      // ring, 7 pairs, q_full, drain
    static constexpr int XCH_OFF = BAR_OFF + NBARS * 8 + 16;
    // per item (two buffers): the slice sums and the max
    static constexpr int XCH_BYTES = 2 * (NSM + 1) * MAXR * 4;
    static constexpr int EPI_STRIDE = 32 * 4 + 16;      // staged O row: 32 floats + pad
    static constexpr size_t SMEM = 1024 + size_t(XCH_OFF) + XCH_BYTES + MAXR * EPI_STRIDE +
                                   NST * 4 + (MAX_BATCH + 1) * 4 + 2 * MAX_BATCH * 4 +
                                   MAX_BATCH + 64;
    static constexpr int S_COL = 0;                     // S buffers: columns [0,64), [64,128)
    static constexpr int O_COL = 2 * PAGE;              // O buffers (by item): D columns each
    static_assert(NST * STAGE_BYTES >= MMA_M * 128, "MMA over-reads must stay in the ring");
    static_assert(O_COL + 2 * D <= TMEM_COLS, "tensor memory columns");
    static_assert(RING_OFF % 1024 == 0 && BAR_OFF % 1024 == 0, "1024-byte aligned buffers");
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

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
                    int chunk_log2, unsigned int* __restrict__ cnt, unsigned int* err) {
    using C = Cfg<D>;
    const int chunk = 1 << chunk_log2;         // keys per work item (CHUNK when invariant)
    const int chunk_pages = chunk / PAGE;
    constexpr int NST = C::NST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sP = smem + C::Q_BYTES;                    // two P buffers
    uint8_t* sStage = smem + C::RING_OFF;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + NST;
    uint64_t* s_full = empty + NST;    // scores of page g in S buffer g&1
    uint64_t* s_empty = s_full + 2;    // ... read by all softmax warps
    uint64_t* p_full = s_empty + 2;    // P of page g in P buffer g&1 (all softmax warps)
    uint64_t* p_empty = p_full + 2;    // P V of page g has completed (MMA commit)
    uint64_t* o_full = p_empty + 2;    // item k's O (buffer k&1) is complete (MMA commit)
    uint64_t* o_empty = o_full + 2;    // ... and read out by the epilogue warp
    uint64_t* xs_bar = o_empty + 2;    // item k's row sums and max are in x_sum[k&1]
    uint64_t* q_full = xs_bar + 2;
    uint64_t* drain = q_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    float* x_sum = reinterpret_cast<float*>(smem + C::XCH_OFF);  // [2][NSM+1][MAXR]
    uint8_t* epi_stage = reinterpret_cast<uint8_t*>(x_sum + 2 * (NSM + 1) * MAXR);
    int* stage_valid = reinterpret_cast<int*>(epi_stage + MAXR * C::EPI_STRIDE);
    int* prefix = stage_valid + NST;  // [B+1]
    int* seq_len = prefix + MAX_BATCH + 1;   // per sequence: length, first token, block width
    int* seq_t0 = seq_len + MAX_BATCH;
    uint8_t* seq_qb = reinterpret_cast<uint8_t*>(seq_t0 + MAX_BATCH);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(seq_qb + MAX_BATCH);
    const unsigned long long wait_ns = wait_budget_ns(err);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv;

    if (warp == MMA_WARP) {  // the MMA warp owns the tensor memory
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    // No griddepcontrol.wait here.  The grid right before this one is always the call's
    // own counter reset, which waits for its predecessors before it lets this grid launch:
    // every kernel that wrote an input (Q, the cache, the block table, the lengths) or
    // last read the workspace has completed by now.  Only the item counters the reset
    // zeroes are not yet safe; the epilogue warp waits for the reset grid before its first
    // count, and triggers the merge's launch after that wait.
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);   // released by the MMA warp's commit after P V
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], NSM);
            mbar_init(&p_full[i], NSM);
            mbar_init(&p_empty[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 1);
            mbar_init(&xs_bar[i], NSM);
        }
        mbar_init(q_full, NSM);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // work items per sequence: chunks x KV heads (0 for a malformed sequence)
    // (kept in shared memory: every warp decodes every item from them)
    for (int b = tid; b < B; b += THREADS) {
        const SeqInfo si = seq_info(seq_lens, cu_q, b);
        const bool ok = seq_ok(si, max_q, max_seq_len, total_q);
        if (!ok) latch_error(err, kErrDeviceArg);
        prefix[b + 1] = ok ? ((si.L + chunk - 1) >> chunk_log2) * Hkv : 0;
        seq_len[b] = si.L;
        seq_t0[b] = si.t0;
        seq_qb[b] = uint8_t(ok ? si.qb : 0);  // <= BI_ATTN_MAX_Q
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
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
    const uint32_t tmem_base = *tmem_slot;

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
    auto seq_of = [&](int b) {
        SeqInfo si;
        si.L = seq_len[b];
        si.t0 = seq_t0[b];
        si.qb = seq_qb[b];
        return si;
    };
    auto pages_of = [&](const SeqInfo& si, int c) {
        return min(chunk_pages, (si.L - c * chunk + PAGE - 1) / PAGE);
    };
    auto give_up = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            latch_error(err, kErrTimeout);
        }
    };
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (ok && !mbar_wait_warp(bar, parity, abort_flag, wait_ns)) ok = false;
        return ok;
    };

    if (warp == PRODUCER) {
        // ------------------------------------------------------------------ producer
        // The whole warp runs the loop (converged, warp-uniform state); one elected lane
        // reads the page index and issues the copies.
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        // K and V are read once per call: first in line for L2 eviction, so the chunk
        // partials (written here, read back by the merge) stay in L2
        const uint64_t kv_policy = l2_policy_evict_first();
        uint32_t g = 0;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
            int b, c, h;
            decode(w, b, c, h);
            const int npages = pages_of(seq_of(b), c);
            int phys_l = -1;  // lane k: the physical page of page (i & ~31) + k of the item
            for (int i = 0; i < npages; ++i, ++g) {
                // the item's block-table entries are read 32 at a time, one per lane, before
                // the wait for a free stage: one load latency per item at the ring's start
                // instead of one per page
                if ((i & 31) == 0) {
                    const int pidx = c * chunk_pages + i + lane;
                    phys_l = (i + lane < npages && pidx < max_pages)
                                 ? block_table[int64_t(b) * max_pages + pidx]
                                 : -1;
                }
                const int s = int(g % NST);
                if (!wait(&empty[s], ((g / NST) & 1u) ^ 1u)) break;
                const int phys = __shfl_sync(0xffffffffu, phys_l, i & 31);
                if (elect_one()) {
                    const bool valid = phys >= 0 && phys < num_pages;
                    stage_valid[s] = valid ? 1 : 0;
                    if (valid) {
                        uint8_t* st = sStage + s * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                        const int row = (phys * Hkv + h) * PAGE;
#pragma unroll
                        for (int bx = 0; bx < C::BOXES; ++bx) {
                            tma_load_2d_hint(st + bx * C::BOX_BYTES, &tmap_k, &full[s], bx * 64,
                                             row, kv_policy);
                            tma_load_2d_hint(st + C::PAGE_BYTES + bx * C::BOX_BYTES, &tmap_v,
                                             &full[s], bx * 64, row, kv_policy);
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
            if (lane == 0) give_up();
            // copies already issued land before the CTA exits (bounded)
            for (int k = 1; k <= NST && k <= int(g); ++k) {
                const uint32_t gg = g - k;
                mbar_wait(&full[gg % NST], (gg / NST) & 1u, nullptr, 100000000ull);
            }
        }
    } else if (warp == MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        // S(page) = Q K^T into S buffer (page & 1); O(item) += P V, issued two pages behind
        // S so the softmax of page i overlaps the scores of page i+1.
        constexpr uint32_t idesc_s = umma_idesc_bf16(MMA_M, PAGE, 0, 0);  // K K-major
        // V N-major; one instruction spans every 64-column box of V (the boxes sit the
        // descriptor's leading-byte offset apart), so each P slice is read once per step
        constexpr uint32_t idesc_pv = umma_idesc_bf16(MMA_M, D, 0, 1);
        const uint64_t q_desc0 = umma_smem_desc(smem_addr(sQ), 16, 1024, 2);
        const uint64_t p_desc0 = umma_smem_desc(smem_addr(sP), 16, 1024, 2);
        const uint64_t k_desc0 = umma_smem_desc(smem_addr(sStage), 16, 1024, 2);
        const uint64_t v_desc0 =
            umma_smem_desc(smem_addr(sStage + C::PAGE_BYTES), C::BOX_BYTES, 1024, 2);
        auto issue_pv = [&](uint32_t gj, int item, bool first, bool last) {
            const int s = int(gj % NST), pb = int(gj & 1u), ob = item & 1;
            if (!wait(&p_full[pb], (gj >> 1) & 1u)) return;
            // the O buffer of this item was read out for item-2
            if (first && !wait(&o_empty[ob], (uint32_t(item >> 1) & 1u) ^ 1u)) return;
            tc_fence_after_sync();
            if (elect_one()) {
                const uint64_t p_desc = p_desc0 + uint64_t((pb * C::P_BYTES) >> 4);
                const uint64_t v_desc = v_desc0 + uint64_t((s * C::STAGE_BYTES) >> 4);
                const uint32_t o_tmem = tmem_base + uint32_t(C::O_COL + ob * D);
#pragma unroll
                for (int k = 0; k < PAGE / 16; ++k)      // keys 16k .. 16k+15: +32 B in P,
                    tc_mma_bf16(o_tmem, p_desc + uint64_t(k * 2),   // +16 rows (2 KB) in V
                                v_desc + uint64_t(k * 128), idesc_pv, (first && k == 0) ? 0u : 1u);
                tc_commit(&p_empty[pb]);
                tc_commit(&empty[s]);   // K and V of the page are no longer read
                if (last) tc_commit(&o_full[ob]);
            }
            __syncwarp();
        };
        // One stream over every page of every item of this CTA: S of page g, then P V of
        // page g-2 (two behind measured 4-5% faster than one behind at large batch: the
        // scores of page g+1 are ready before the softmax finishes page g), and the next
        // item's first scores are computed while the softmax finishes the previous item
        // (its Q is published early, see the softmax warps).
        uint32_t g = 0;
        int item = 0;
        struct Pend {
            int item;
            bool first, last;
        };
        Pend pa{0, false, false}, pb{0, false, false};  // pending P V products, pa oldest
        int npend = 0;
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++item) {
            int b, c, h;
            decode(w, b, c, h);
            const int npages = pages_of(seq_of(b), c);
            if (!wait(q_full, uint32_t(item) & 1u)) break;
            for (int i = 0; i < npages; ++i) {
                const uint32_t gi = g + uint32_t(i);
                const int s = int(gi % NST), sb = int(gi & 1u);
                if (!wait(&full[s], (gi / NST) & 1u) || !wait(&s_empty[sb], ((gi >> 1) & 1u) ^ 1u))
                    break;
                tc_fence_after_sync();
                if (elect_one()) {
                    const uint64_t k_desc = k_desc0 + uint64_t((s * C::STAGE_BYTES) >> 4);
                    const uint32_t d = tmem_base + uint32_t(C::S_COL + sb * PAGE);
#pragma unroll
                    for (int bx = 0; bx < C::BOXES; ++bx)      // head dims 64bx .. 64bx+63
#pragma unroll
                        for (int k = 0; k < 4; ++k)            // in 16-wide steps: +32 B
                            tc_mma_bf16(d, q_desc0 + uint64_t(bx * (C::QBOX_BYTES >> 4) + k * 2),
                                        k_desc + uint64_t(bx * (C::BOX_BYTES >> 4) + k * 2),
                                        idesc_s, (bx | k) != 0 ? 1u : 0u);
                    tc_commit(&s_full[sb]);
                }
                __syncwarp();
                if (npend == PV_LAG) {
                    issue_pv(gi - uint32_t(PV_LAG), pa.item, pa.first, pa.last);
                    pa = pb;
                    --npend;
                }
                if (!ok) break;
                const Pend cur{item, i == 0, i == npages - 1};
                if (npend == 0) pa = cur; else pb = cur;
                ++npend;
            }
            g += uint32_t(npages);
        }
        if (ok && npend >= 1) issue_pv(g - uint32_t(npend), pa.item, pa.first, pa.last);
        if (ok && npend == 2) issue_pv(g - 1u, pb.item, pb.first, pb.last);
        if (!ok && lane == 0) give_up();
        // every MMA this warp issued completes before tensor memory is released
        if (elect_one()) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, nullptr, 100000000ull);
    } else if (warp == EPILOGUE) {
        // ------------------------------------------------------------------ epilogue
        // Item k's O (tensor-memory lanes 0..31, buffer k&1) and its row sums and max,
        // written as the chunk partial (m, l, o) of every row that sees the chunk.  The
        // softmax warps move on to the next item meanwhile.
        const int r = lane;
        int item = 0;
        bool reset_done = false;  // griddepcontrol.wait passed (the counters are zeroed)
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++item) {
            int b, c, h;
            decode(w, b, c, h);
            const SeqInfo si = seq_of(b);
            const int R = si.qb * G;
            const int j = r / G, gg = r - (r / G) * G;
            const int pos = r < R ? si.L - si.qb + j : -1;
            const int ob = item & 1;
            const uint32_t par = uint32_t(item >> 1) & 1u;
            if (!wait(&xs_bar[ob], par) || !wait(&o_full[ob], par)) break;
            tc_fence_after_sync();
            const float* xs = x_sum + ob * ((NSM + 1) * MAXR);
            const float l_tot = ((xs[r] + xs[MAXR + r]) + xs[2 * MAXR + r]) + xs[3 * MAXR + r];
            const float m_ref = xs[NSM * MAXR + r];
            const bool store = r < R && pos >= c * chunk;
            const int64_t idx = (int64_t(si.t0 + j) * Hq + int64_t(h) * G + gg) * maxC + c;
            // O row r of 32 columns at a time: staged through shared memory (rows padded
            // to 144 B, conflict-free) so that each store instruction writes four rows'
            // 128-byte segments instead of 32 scattered 16-byte pieces
            const int rr = lane >> 3, part = lane & 7;  // reader: row within 4, 16-B piece
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t v[32];
                tmem_load_32x32b_x32_sync(tmem_base + uint32_t(C::O_COL + ob * D + cc * 32), v);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<uint4*>(epi_stage + r * C::EPI_STRIDE + k * 16) =
                        make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < MAXR / 4; ++k) {
                    const int row = 4 * k + rr;
                    const bool st = __shfl_sync(0xffffffffu, store ? 1 : 0, row) != 0;
                    const int64_t ridx = __shfl_sync(0xffffffffu, idx, row);
                    if (st)
                        *reinterpret_cast<uint4*>(ws_o + ridx * D + cc * 32 + part * 4) =
                            *reinterpret_cast<const uint4*>(epi_stage + row * C::EPI_STRIDE +
                                                           part * 16);
                }
                __syncwarp();
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[ob]);
            if (store) *reinterpret_cast<float2*>(ws_ml + idx * 2) = make_float2(m_ref, l_tot);
            // the item's partials are written: count it for its (sequence, KV head), which
            // the merge waits on (every lane's stores are ordered before the count)
            __threadfence();
            __syncwarp();
            if (!reset_done) {
                pdl_wait();
                pdl_trigger();
                reset_done = true;
            }
            if (lane == 0) atomicAdd(cnt + b * Hkv + h, 1u);
        }
        if (!ok && lane == 0) give_up();
        // a CTA with no item (or one that gave up) still waits before it completes, so the
        // merge grid never launches ahead of the reset
        if (!reset_done) {
            pdl_wait();
            pdl_trigger();
        }
    } else if (warp < NSM) {
        // ------------------------------------------------------------------- softmax
        // Warp sw (0..3) reads tensor-memory lanes 32sw .. 32sw+31, which hold a copy of
        // the query rows (row r = lane, so each warp sees every score of the row), and
        // owns keys 16sw .. 16sw+15 of every page: its slice of each P row, its slice of
        // the row sum.  The four warps compute the same reference max m, so their P
        // slices form one P row and one MMA accumulates the whole O in lanes 0..31.
        const int sw = warp;
        const int r = lane;
        uint32_t g = 0;
        int item = 0;
        int q_b = -1, q_h = -1;  // (sequence, KV head) whose Q tile sQ holds
        const uint32_t lane_base = uint32_t(32 * sw) << 16;
        // Q tile of item w, (b, h): rows 32sw + r hold query row r = j*G + gg (zero past
        // R); rewritten only when (b, h) changes.  Item w+grid's tile is published as
        // soon as this warp has read the scores of item w's last page: every MMA that
        // read the old tile has completed by then.
        auto publish_q = [&](int wq) {
            if (wq < total) {
                int b, c, h;
                decode(wq, b, c, h);
                if (b != q_b || h != q_h) {
                    const SeqInfo si = seq_of(b);
                    const int R = si.qb * G;
                    const int j = r / G, gg = r - (r / G) * G;
                    const __nv_bfloat16* src =
                        q + (int64_t(si.t0 + j) * Hq + int64_t(h) * G + gg) * D;
#pragma unroll
                    for (int ch = 0; ch < D / 8; ++ch) {
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (r < R) v = *reinterpret_cast<const uint4*>(src + ch * 8);
                        *reinterpret_cast<uint4*>(sQ + (ch >> 3) * C::QBOX_BYTES +
                                                  swz(32 * sw + r, ch & 7)) = v;
                    }
                    q_b = b;
                    q_h = h;
                    fence_proxy_async_smem();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);  // one arrival per item (also the last)
        };
        publish_q(blockIdx.x);
        for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++item) {
            int b, c, h;
            decode(w, b, c, h);
            const SeqInfo si = seq_of(b);
            const int L = si.L, qb = si.qb;
            const int npages = pages_of(si, c);
            const int R = qb * G;
            const int pos = r < R ? L - qb + r / G : -1;
            const int ob = item & 1;

            float m_ref = -INFINITY, l_run = 0.f;
            for (int i = 0; i < npages && ok; ++i) {
                const uint32_t gi = g + uint32_t(i);
                const int s = int(gi % NST), sb = int(gi & 1u);
                const uint32_t par = (gi >> 1) & 1u;
                const int page0 = c * chunk + i * PAGE;  // first key of the page
                // the whole page of scores of row r (every lane quarter holds all 64 keys
                // of the query rows) and this warp's 16-key slice of it, then release the
                // S buffer
                if (!wait(&s_full[sb], par)) break;
                tc_fence_after_sync();
                uint32_t sa[PAGE], sv[KSL];
                const uint32_t s_tm = tmem_base + lane_base + uint32_t(C::S_COL + sb * PAGE);
                tmem_load_x64_x16_sync(s_tm, s_tm + uint32_t(sw * KSL), sa, sv);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                if (i == npages - 1) publish_q(w + gridDim.x);
                // the stage's K/V landed before its scores were computed; this wait only
                // orders the valid flag and the V rows zeroed below after the copy
                if (!wait(&full[s], (gi / NST) & 1u)) break;
                const bool valid = stage_valid[s] != 0;

                // causal mask (masked keys -> -inf) and the row max over the page, taken on
                // the raw scores (exact: max does not round, so neither the tree nor its
                // grouping matters, and each warp finds the same page max with no exchange);
                // scaling by the positive scale_log2 afterwards gives the max of the scaled
                // scores.  A page that every query of the block sees in full needs no mask
                // for the block's rows; the padding rows past R (zero Q, never stored) then
                // see it too, which changes nothing in the other rows.
                float sl[KSL], m_raw;
                {
                    float a[PAGE];
                    if (valid && page0 + PAGE - 1 <= L - qb) {
#pragma unroll
                        for (int k = 0; k < PAGE; ++k) a[k] = __uint_as_float(sa[k]);
#pragma unroll
                        for (int k = 0; k < KSL; ++k) sl[k] = __uint_as_float(sv[k]);
                    } else {
                        const int lim = valid ? pos - page0 : -1;  // last visible key, or < 0
#pragma unroll
                        for (int k = 0; k < PAGE; ++k)
                            a[k] = k <= lim ? __uint_as_float(sa[k]) : -INFINITY;
#pragma unroll
                        for (int k = 0; k < KSL; ++k)
                            sl[k] = sw * KSL + k <= lim ? __uint_as_float(sv[k]) : -INFINITY;
                    }
                    float t1[22], t2[8];
#pragma unroll
                    for (int k = 0; k < 21; ++k) t1[k] = fmax3(a[3 * k], a[3 * k + 1], a[3 * k + 2]);
                    t1[21] = a[63];
#pragma unroll
                    for (int k = 0; k < 7; ++k) t2[k] = fmax3(t1[3 * k], t1[3 * k + 1], t1[3 * k + 2]);
                    t2[7] = t1[21];
                    m_raw = fmax3(fmax3(t2[0], t2[1], t2[2]), fmax3(t2[3], t2[4], t2[5]),
                                  fmaxf(t2[6], t2[7]));
                }
                const float m_page = m_raw * scale_log2;

                // reference max: raised (and O, l rescaled) only when the page max exceeds
                // it by more than 2^8, so p = exp2(s - m_ref) <= 2^8
                const bool raise = m_page > m_ref + kRescaleLog2 ||
                                   (m_ref == -INFINITY && m_page != -INFINITY);
                const float factor = raise ? ex2(m_ref - m_page) : 1.f;  // 0 on the first
                if (raise) m_ref = m_page;
                l_run *= factor;
                // this warp's 16 keys; a masked key (-inf) gives p = +0
                // p = exp2(s * scale_log2 - m), the row-slice sum by a fixed pairwise tree
                float pv[KSL];
                {
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
                    for (int k = 0; k < KSL; ++k) pv[k] = ex2(fmaf(sl[k], scale_log2, -m_use));
                }
                uint32_t pk[KSL / 2];
#pragma unroll
                for (int k = 0; k < KSL; k += 2) pk[k / 2] = pack_bf16x2(pv[k], pv[k + 1]);
#pragma unroll
                for (int width = KSL / 2; width >= 1; width /= 2)
#pragma unroll
                    for (int k = 0; k < width; ++k) pv[k] = pv[k] + pv[k + width];
                const float ps = pv[0];
                l_run = l_run + ps;
                // P buffer sb is free once P V of page gi-2 has completed
                if (!wait(&p_empty[sb], par ^ 1u)) break;
                if (sw == 0 && i > 0 && __any_sync(0xffffffffu, raise)) {
                    // O (lanes 0..31) *= factor after P V of page gi-1 has completed
                    const uint32_t gp = gi - 1u;
                    if (!wait(&p_empty[gp & 1u], (gp >> 1) & 1u)) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t v[32];
                        const uint32_t ta = tmem_base + uint32_t(C::O_COL + ob * D + cc * 32);
                        tmem_load_32x32b_x32_sync(ta, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            v[k] = __float_as_uint(__uint_as_float(v[k]) * factor);
                        tmem_store_32x32b_x32_sync(ta, v);
                    }
                    tc_fence_before_sync();
                }
                // this warp's 16 keys of P row r (two 16-byte pieces of the 128-byte row)
                uint8_t* pbuf = sP + sb * C::P_BYTES;
                *reinterpret_cast<uint4*>(pbuf + swz(r, 2 * sw)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(pbuf + swz(r, 2 * sw + 1)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
                // V rows of this slice past the sequence end (or of an invalid page) are
                // zeroed so unwritten cache slots cannot inject NaN/Inf through 0 * v
                const int vend = valid ? L - page0 : 0;  // first row to zero
                if (vend < (sw + 1) * KSL) {
                    const int r0 = max(vend, sw * KSL);
                    uint8_t* vst = sStage + s * C::STAGE_BYTES + C::PAGE_BYTES;
                    const int n16 = ((sw + 1) * KSL - r0) * 8;  // 16-byte pieces per box
                    for (int idx = lane; idx < C::BOXES * n16; idx += 32) {
                        const int bx = idx / n16, rem = idx - bx * n16;
                        *reinterpret_cast<uint4*>(vst + bx * C::BOX_BYTES + r0 * 128 + rem * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
            }
            if (!ok) break;
            g += uint32_t(npages);
            // the slice sums (and the shared max) for the epilogue warp, once it has read
            // this buffer's previous contents (item-2)
            if (!wait(&o_empty[ob], (uint32_t(item >> 1) & 1u) ^ 1u)) break;
            float* xs = x_sum + ob * ((NSM + 1) * MAXR);
            xs[sw * MAXR + r] = l_run;
            if (sw == 0) xs[NSM * MAXR + r] = m_ref;
            __syncwarp();
            if (lane == 0) mbar_arrive(&xs_bar[ob]);
        }
        if (!ok && lane == 0) give_up();
    }
    // every warp is done with tensor memory and shared memory past this barrier
    tc_fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// --------------------------------------------------------------------- merge kernel

constexpr int MERGE_WARPS = 8;    // chunk ranges of the merge tree
constexpr int64_t kMergeRowsMin = 4096;  // rows from which a warp per row merges
constexpr int MERGE_UNROLL = 17;  // partials requested per round trip (136 chunks in 8)

// The merge tree of one (token, query head) row with nC = pos/chunk + 1 chunk partials:
// range w = [w*nC/8, (w+1)*nC/8) is folded in ascending chunk order (its max first, then
// the exp2-weighted sums), and the eight range results are combined in ascending range
// order -- a tree fixed by nC, i.e. by the query's position.  Both merge kernels below run
// exactly these two functions, so they give the same bits.

// Fold chunks [c0, c1) of the row at `base` (lane holds dims lane*PER ..): range max Mw,
// weighted sum Lw and weighted o sums acc.
template <int D>
__device__ __forceinline__ void merge_fold(const float* __restrict__ ws_o,
                                           const float* __restrict__ ws_ml, int64_t base, int c0,
                                           int c1, int lane, float& Mw, float& Lw,
                                           float (&acc)[D / 32]) {
    constexpr int PER = D / 32;
    // The first MERGE_UNROLL partials of the range are requested before anything else
    // (for ranges up to MERGE_UNROLL chunks: all of them, in one global round trip).
    // loads at L2 (ld.global.cg): the partial kernel may still be running, and this SM's
    // L1 may hold a neighbouring row's line from before that row was complete
    auto load = [&](int c, float (&v)[PER], float2& ml) {
        ml = __ldcg(reinterpret_cast<const float2*>(ws_ml + (base + c) * 2));
        const float* src = ws_o + (base + c) * D + lane * PER;
        if (PER == 4) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(src));
            v[0] = f.x; v[1 % PER] = f.y; v[2 % PER] = f.z; v[3 % PER] = f.w;
        } else {
            const float2 f = __ldcg(reinterpret_cast<const float2*>(src));
            v[0] = f.x; v[1 % PER] = f.y;
        }
    };
    float v[MERGE_UNROLL][PER];
    float2 ml[MERGE_UNROLL];
#pragma unroll
    for (int u = 0; u < MERGE_UNROLL; ++u)
        if (c0 + u < c1) load(c0 + u, v[u], ml[u]);

    // range max (exact in any order): from the registers when the whole range was loaded
    // above, else lanes stride over the chunks and a butterfly combines them
    Mw = -INFINITY;
    if (c1 - c0 <= MERGE_UNROLL) {
#pragma unroll
        for (int u = 0; u < MERGE_UNROLL; ++u)
            if (c0 + u < c1) Mw = fmaxf(Mw, ml[u].x);
    } else {
        for (int c = c0 + lane; c < c1; c += 32) Mw = fmaxf(Mw, __ldcg(ws_ml + (base + c) * 2));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, off));
    }

    Lw = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int c = c0; c < c1; c += MERGE_UNROLL) {
        if (c > c0) {
#pragma unroll
            for (int u = 0; u < MERGE_UNROLL; ++u)  // issue the loads of the next chunks first
                if (c + u < c1) load(c + u, v[u], ml[u]);
        }
#pragma unroll
        for (int u = 0; u < MERGE_UNROLL; ++u) {  // then fold them in ascending chunk order
            if (c + u < c1) {
                const float wgt = exp2f(ml[u].x - Mw);
                Lw = Lw + wgt * ml[u].y;
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] = acc[i] + wgt * v[u][i];
            }
        }
    }
}

// Combine the eight range results (Mw[w], Lw[w], acc of range w through get_acc(w, i)) in
// ascending range order and store the row (and its natural-log LSE).
template <int D, class AccFn>
__device__ __forceinline__ void merge_combine(const float (&Mw)[MERGE_WARPS],
                                              const float (&Lw)[MERGE_WARPS], AccFn get_acc,
                                              int lane, __nv_bfloat16* __restrict__ dst_row,
                                              float* lse_slot) {
    constexpr int PER = D / 32;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) M = fmaxf(M, Mw[w]);
    float L = 0.f;
    float o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = 0.f;
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) {
        const float wgt = exp2f(Mw[w] - M);  // an empty range has Mw = -inf: weight 0
        L = L + wgt * Lw[w];
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = o[i] + wgt * get_acc(w, i);
    }
    __nv_bfloat16* dst = dst_row + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[i] = __float2bfloat16_rn(o[i] / L);
    if (lse_slot && lane == 0) *lse_slot = (M + log2f(L)) * kLn2;
}

// Row (token t, query head hq) of the call: its sequence and position, or false when the
// sequence is malformed or the token belongs to none.
__device__ __forceinline__ bool merge_row(const int32_t* __restrict__ seq_lens,
                                          const int32_t* __restrict__ cu_q, int B, int total_q,
                                          int max_q, int max_seq_len, int t, int& pos, int& bq,
                                          int& len) {
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
    if (!seq_ok(si, max_q, max_seq_len, total_q) || t < si.t0 || t >= si.t0 + si.qb) return false;
    pos = si.L - si.qb + (t - si.t0);
    bq = b;
    len = si.L;
    return true;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits (bounded by timeout_ns) until the partial kernel has counted `target` finished
// items of one (sequence, KV head); acquire, so the items' partials are visible to this
// thread and, after a barrier, to its CTA or warp.  False on timeout.
__device__ __noinline__ bool wait_items(const unsigned int* cnt, unsigned int target,
                                        unsigned long long timeout_ns) {
    if (ld_acquire_u32(cnt) >= target) return true;
    const long long budget = static_cast<long long>(timeout_ns) * 5 / 2;  // cycles
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(256);
        if (ld_acquire_u32(cnt) >= target) return true;
        if (clock64() - t0 > budget) return false;
    }
}

// Zeroes the item counters of one call (after the previous grid in the stream, which may
// be the previous call's merge still reading them); the partial kernel waits for this grid.
__global__ void __launch_bounds__(256) attn_count_reset_kernel(unsigned int* cnt, int n) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256) cnt[i] = 0u;
}

// One CTA per row: warp w folds range w (latency: a few rows, long contexts).
template <int D>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
attn_merge_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
                  int total_q, int max_q, int max_seq_len, int Hq, int Hkv,
                  const float* ws_o, const float* ws_ml, int maxC, int chunk_log2,
                  const unsigned int* cnt, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, unsigned int* err) {
    constexpr int PER = D / 32;
    __shared__ float sM[MERGE_WARPS], sL[MERGE_WARPS];
    __shared__ float sO[MERGE_WARPS][D];
    __shared__ int s_ready;
    // With item counters this grid may start while the partial kernel runs: every grid
    // before that kernel has completed (it waited for them before letting this one
    // launch), and each row waits for its own (sequence, KV head)'s items below.
    // Without counters, the whole previous grid.
    if (!cnt) pdl_wait();
    pdl_trigger();
    const int t = int(blockIdx.x / unsigned(Hq));
    const int hq = int(blockIdx.x - unsigned(t) * unsigned(Hq));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int pos, b, L;
    if (!merge_row(seq_lens, cu_q, B, total_q, max_q, max_seq_len, t, pos, b, L)) return;
    if (cnt) {
        if (threadIdx.x == 0) {
            const unsigned int items = unsigned((L + (1 << chunk_log2) - 1) >> chunk_log2);
            s_ready = wait_items(cnt + b * Hkv + hq / (Hq / Hkv), items, wait_budget_ns(err)) ? 1 : 0;
            if (!s_ready) latch_error(err, kErrTimeout);
        }
        __syncthreads();
        if (!s_ready) return;
    }
    const int nC = (pos >> chunk_log2) + 1;
    const int64_t base = (int64_t(t) * Hq + hq) * maxC;
    float Mw, Lw, acc[PER];
    merge_fold<D>(ws_o, ws_ml, base, warp * nC / MERGE_WARPS, (warp + 1) * nC / MERGE_WARPS,
                  lane, Mw, Lw, acc);
    if (lane == 0) {
        sM[warp] = Mw;
        sL[warp] = Lw;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) sO[warp][lane * PER + i] = acc[i];
    __syncthreads();
    if (warp != 0) return;
    float M8[MERGE_WARPS], L8[MERGE_WARPS];
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) {
        M8[w] = sM[w];
        L8[w] = sL[w];
    }
    merge_combine<D>(M8, L8, [&](int w, int i) { return sO[w][lane * PER + i]; }, lane,
                     out + (int64_t(t) * Hq + hq) * D, lse ? lse + int64_t(t) * Hq + hq : nullptr);
}

// One warp per row, eight rows per CTA: the same tree, its eight ranges folded one after
// another (throughput: many rows, e.g. a prefill block).  UNR (>= the rows' chunk count)
// sizes the register window that holds a row's partials: the smaller it is, the more CTAs
// share an SM and the more rows' loads are in flight (it changes no arithmetic).
template <int D, int UNR>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
attn_merge_rows_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q,
                       int B, int total_q, int max_q, int max_seq_len, int Hq, int Hkv,
                       const float* ws_o, const float* ws_ml, int maxC, int chunk_log2,
                       const unsigned int* cnt, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse, unsigned int* err) {
    constexpr int PER = D / 32;
    if (!cnt) pdl_wait();  // see attn_merge_kernel
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * MERGE_WARPS + warp;
    if (row >= int64_t(total_q) * Hq) return;
    const int t = int(row / Hq);
    const int hq = int(row - int64_t(t) * Hq);
    int pos, b, L;
    if (!merge_row(seq_lens, cu_q, B, total_q, max_q, max_seq_len, t, pos, b, L)) return;
    if (cnt) {
        int ready = 1;
        if (lane == 0) {
            const unsigned int items = unsigned((L + (1 << chunk_log2) - 1) >> chunk_log2);
            ready = wait_items(cnt + b * Hkv + hq / (Hq / Hkv), items, wait_budget_ns(err)) ? 1 : 0;
            if (!ready) latch_error(err, kErrTimeout);
        }
        __syncwarp();  // orders lane 0's acquire before the other lanes' loads
        if (!__shfl_sync(0xffffffffu, ready, 0)) return;
    }
    const int nC = (pos >> chunk_log2) + 1;
    const int64_t base = (int64_t(t) * Hq + hq) * maxC;
    // the host picks UNR >= maxC >= nC for every valid row
    if (nC > UNR) return;
    float M8[MERGE_WARPS], L8[MERGE_WARPS], acc8[MERGE_WARPS][PER];
    // every partial of the row in one round trip, then each range folded from the
    // registers with merge_fold's arithmetic (max first, then the weighted sums in
    // ascending chunk order)
    float v[UNR][PER];
    float2 ml[UNR];
#pragma unroll
    for (int c = 0; c < UNR; ++c) {
        if (c < nC) {  // at L2, as merge_fold loads
            ml[c] = __ldcg(reinterpret_cast<const float2*>(ws_ml + (base + c) * 2));
            const float* src = ws_o + (base + c) * D + lane * PER;
            if (PER == 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(src));
                v[c][0] = f.x; v[c][1 % PER] = f.y; v[c][2 % PER] = f.z; v[c][3 % PER] = f.w;
            } else {
                const float2 f = __ldcg(reinterpret_cast<const float2*>(src));
                v[c][0] = f.x; v[c][1 % PER] = f.y;
            }
        }
    }
#pragma unroll
    for (int w = 0; w < MERGE_WARPS; ++w) {
        const int c0 = w * nC / MERGE_WARPS, c1 = (w + 1) * nC / MERGE_WARPS;
        float Mw = -INFINITY;
#pragma unroll
        for (int c = 0; c < UNR; ++c)
            if (c >= c0 && c < c1) Mw = fmaxf(Mw, ml[c].x);
        float Lw = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc8[w][i] = 0.f;
#pragma unroll
        for (int c = 0; c < UNR; ++c) {
            if (c >= c0 && c < c1) {
                const float wgt = exp2f(ml[c].x - Mw);
                Lw = Lw + wgt * ml[c].y;
#pragma unroll
                for (int i = 0; i < PER; ++i) acc8[w][i] = acc8[w][i] + wgt * v[c][i];
            }
        }
        M8[w] = Mw;
        L8[w] = Lw;
    }
    merge_combine<D>(M8, L8, [&](int w, int i) { return acc8[w][i]; }, lane,
                     out + (int64_t(t) * Hq + hq) * D, lse ? lse + int64_t(t) * Hq + hq : nullptr);
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

// Workspace of one call: the chunk partials (o [T][Hq][chunks][D], then (m, l)
// [T][Hq][chunks][2], fp32), then at the next 16-byte boundary one item counter per
// (sequence, KV head), bounded by T x Hq words.
size_t partials_bytes(int64_t total_q, int64_t hq, int64_t head_dim, int64_t chunks) {
    const size_t b = size_t(total_q) * size_t(hq) * size_t(chunks) * size_t(head_dim + 2) *
                     sizeof(float);
    return (b + 15) / 16 * 16;
}

size_t workspace_for(int64_t total_q, int64_t hq, int64_t head_dim, int64_t max_seq_len,
                     int chunk_log2) {
    const int64_t chunk = int64_t(1) << chunk_log2;
    const int64_t chunks = (max_seq_len + chunk - 1) / chunk;
    return partials_bytes(total_q, hq, head_dim, chunks) +
           (size_t(total_q) * size_t(hq) * sizeof(unsigned int) + 15) / 16 * 16;
}
template <int D>
cudaError_t launch_attention_t(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                               float scale, void* out, float* lse, void* workspace,
                               int chunk_log2, cudaStream_t stream) {
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
    const int chunk = 1 << chunk_log2;
    const int maxC = int((a.max_seq_len + chunk - 1) / chunk);
    const int64_t items_bound = a.batch * int64_t(maxC) * a.hkv;
    if (items_bound > 0x7fffffffLL) return cudaErrorNotSupported;
    const int grid = int(items_bound < dev.num_sms ? items_bound : dev.num_sms);
    float* ws_o = static_cast<float*>(workspace);
    float* ws_ml = ws_o + a.total_q * a.hq * int64_t(maxC) * D;
    unsigned int* cnt = reinterpret_cast<unsigned int*>(
        static_cast<uint8_t*>(workspace) + partials_bytes(a.total_q, a.hq, D, maxC));
    const int ncnt = int(a.batch * a.hkv);
    const float scale_log2 = scale * kLog2e;
    cudaError_t e = launch_pdl(attn_count_reset_kernel, dim3((ncnt + 1023) / 1024), dim3(256), 0,
                               stream, cnt, ncnt);
    if (e != cudaSuccess) return e;
    e = launch_pdl(
        kern, dim3(grid), dim3(THREADS), Cf::SMEM, stream, tk, tv,
        static_cast<const __nv_bfloat16*>(q), a.block_table, int(a.max_pages), int(a.num_pages),
        a.seq_lens, a.cu_q, int(a.batch), int(a.total_q), int(a.max_q), int(a.max_seq_len),
        int(a.hq), int(a.hkv), scale_log2, ws_o, ws_ml, maxC, chunk_log2, cnt, dev.err_word);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(a, workspace, chunk_log2, out, lse, cnt, dev.err_word, stream);
}

}  // namespace

cudaError_t launch_attn_merge(const PagedArgs& a, void* workspace, int chunk_log2, void* out,
                              float* lse, const unsigned int* cnt, unsigned int* err,
                              cudaStream_t stream) {
    const int chunk = 1 << chunk_log2;
    const int maxC = int((a.max_seq_len + chunk - 1) / chunk);
    const float* ws_o = static_cast<const float*>(workspace);
    const float* ws_ml = ws_o + a.total_q * a.hq * int64_t(maxC) * a.head_dim;
    const int64_t rows = a.total_q * a.hq;
    // few rows or long rows: a CTA per row, its eight ranges in parallel; many rows of at
    // most MERGE_UNROLL chunks: a warp per row, all its partials loaded at once (both run
    // the same tree, so the choice does not change any bit)
    if (rows < kMergeRowsMin || maxC > MERGE_UNROLL) {
        auto kern = a.head_dim == 64 ? attn_merge_kernel<64> : attn_merge_kernel<128>;
        return launch_pdl(kern, dim3(unsigned(rows)), dim3(MERGE_WARPS * 32), 0, stream,
                          a.seq_lens, a.cu_q, int(a.batch), int(a.total_q), int(a.max_q),
                          int(a.max_seq_len), int(a.hq), int(a.hkv), ws_o, ws_ml, maxC,
                          chunk_log2, cnt, static_cast<__nv_bfloat16*>(out), lse, err);
    }
    auto kern = a.head_dim == 64
                    ? (maxC <= 4 ? attn_merge_rows_kernel<64, 4>
                                 : maxC <= 8 ? attn_merge_rows_kernel<64, 8>
                                             : attn_merge_rows_kernel<64, MERGE_UNROLL>)
                    : (maxC <= 4 ? attn_merge_rows_kernel<128, 4>
                                 : maxC <= 8 ? attn_merge_rows_kernel<128, 8>
                                             : attn_merge_rows_kernel<128, MERGE_UNROLL>);
    return launch_pdl(kern, dim3(unsigned((rows + MERGE_WARPS - 1) / MERGE_WARPS)),
                      dim3(MERGE_WARPS * 32), 0, stream, a.seq_lens, a.cu_q, int(a.batch),
                      int(a.total_q), int(a.max_q), int(a.max_seq_len), int(a.hq), int(a.hkv),
                      ws_o, ws_ml, maxC, chunk_log2, cnt, static_cast<__nv_bfloat16*>(out), lse,
                      err);
}

size_t attn_workspace_bytes(int64_t total_q, int64_t hq, int64_t head_dim, int64_t max_seq_len) {
    return workspace_for(total_q, hq, head_dim, max_seq_len, CHUNK_LOG2);
}

int attn_chunk_log2(const PagedArgs& a, size_t ws_bytes, int num_sms, bool invariant) {
    if (invariant) return CHUNK_LOG2;
    // Non-invariant call: the chunk length that minimises a simple cost in page-times.
    // Sequences are taken to be max_seq_len long.  Work items are dealt round-robin to
    // the persistent CTAs, so the busiest CTA runs ceil(items / SMs) of them; in the
    // worst case only one in every (chunks per sequence) of those is a short last chunk.
    // An item costs its pages plus a fixed overhead (pipeline turn-around, ~half a page)
    // plus its partials (written by the partial kernel, read back by the merge) in
    // page-equivalents of K+V bytes.  Ties go to the longer chunk (fewer partials).
    // Only chunk lengths whose partials fit in the caller's workspace are considered.
    const int64_t group = a.hq / a.hkv;
    const double page_bytes = double(PAGE) * double(a.head_dim) * 2.0 * 2.0;
    const double item_ovh =
        0.5 + double(a.max_q * group) * double(a.head_dim + 2) * 4.0 * 2.0 / page_bytes;
    int best = CHUNK_LOG2;
    double best_cost = -1.0;
    for (int lg = MAX_CHUNK_LOG2; lg >= MIN_CHUNK_LOG2; --lg) {
        if (workspace_for(a.total_q, a.hq, a.head_dim, a.max_seq_len, lg) > ws_bytes) continue;
        const int64_t chunk = int64_t(1) << lg;
        const int64_t chunks = (a.max_seq_len + chunk - 1) / chunk;
        const int64_t items = a.batch * a.hkv * chunks;
        const int64_t per_cta = (items + num_sms - 1) / num_sms;
        const int64_t tails = per_cta / chunks;
        const double full_pages = double(chunk / PAGE);
        const double tail_pages = double((a.max_seq_len - (chunks - 1) * chunk + PAGE - 1) / PAGE);
        const double cost = double(per_cta) * item_ovh + double(per_cta - tails) * full_pages +
                            double(tails) * tail_pages;
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = lg;
        }
    }
    return best;
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
                             int chunk_log2, cudaStream_t stream) {
    if (chunk_log2 < MIN_CHUNK_LOG2 || chunk_log2 > MAX_CHUNK_LOG2) return cudaErrorNotSupported;
    if (a.head_dim == 64)
        return launch_attention_t<64>(dev, q, a, scale, out, lse, workspace, chunk_log2, stream);
    return launch_attention_t<128>(dev, q, a, scale, out, lse, workspace, chunk_log2, stream);
}

}  // namespace bi
