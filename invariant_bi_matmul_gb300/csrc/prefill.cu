// prefill.cu -- chunked-prefill / prefix-cache attention: causal attention of blocks of
// any width over a bf16 paged KV cache, each query reduced exactly as the decode / verify
// kernel (attention.cu) reduces it, so a token's output bits do not depend on how many
// of its predecessors were already cached or on how the prompt was cut into blocks.
//
// Source: book chapter "Batch-invariant kernels: why temperature-0 decoding is still
// nondeterministic", Case 6, Attention row, and the paragraph after the strategy table:
// serving engines slice sequences (chunked prefill, prefix caching), and token 1000 must
// reduce identically whether 0 or 999 tokens are already cached -- the cache and the new
// tokens are scored in one loop, not two.
//
// Per query row (position pos), identical to attention.cu:
//   * chunks of CHUNK keys from key 0; chunk c is reduced by the row only if pos >= c*CHUNK;
//   * per 64-key page: S = Q K^T by tcgen05 (M = 128, N = 64, the head dimension in 16-wide
//     steps, ascending), keys > pos masked to -inf, the exact page row max, the reference
//     max m raised only when the page max exceeds it by more than 2^8 (O and the sums then
//     scaled by 2^(m_old - m_new)), P = 2^(S*scale_log2 - m) rounded to bf16 (both
//     powers by the same ex2 as the decode kernel),
//     O += P V by tcgen05 (N = head_dim, keys in 16-wide steps, ascending), and the row
//     sum kept as four running sums of the page's 16-key slices (each slice summed by the
//     same pairwise tree), added in ascending slice order at the end of the chunk;
//   * the chunk partials (m, l, o) go to the same workspace and through the same merge
//     kernel.
// A chunk's pages run to the sequence's end, as in the decode kernel, whatever the tile.
//
// What differs from the decode kernel is the tile: 128 DIFFERENT query rows (128/G tokens
// x the G query heads of one KV head), one per tensor-memory lane, instead of <= 32 rows
// repeated in each lane quarter.  So each softmax warp owns the 32 rows of its lane
// quarter and all 64 keys of a page (no exchange of slice maxima), and four epilogue
// warps, one per quarter, write the partials.
//
// Warps: 0..3 softmax, 4..7 epilogue (quarter = warp mod 4), 8 TMA producer of K/V pages,
// 9 S issuer (and TMEM owner; it also copies each item's Q tile by TMA), 10 P V issuer.
// The two issuers run apart, so the scores of later pages are never queued behind a P V
// that waits for its P, and P has four tensor-memory buffers, so the softmax of page g
// waits only for the P V of page g-4.  Work items
// (sequence, query tile, KV head, chunk), chunk fastest, are dealt to CTAs in contiguous
// runs so that consecutive items share the Q tile.
#include "attn_common.cuh"

namespace bi {
namespace {

constexpr int P_NSM = 4;                 // softmax warps
constexpr int P_EPI = 4;                 // first epilogue warp (quarters 0..3)
constexpr int P_PRODUCER = 8, P_MMA = 9, P_PV = 10;
constexpr int P_THREADS = 11 * 32;
constexpr int P_NPB = 4;                 // P buffers in tensor memory (by page)
static_assert(PAGE == 64, "the page max below is a three-input max tree over 64 keys");
constexpr int P_ROWS = 128;              // query rows per tile, one per TMEM lane
constexpr int P_TMEM_COLS = 512;
constexpr int P_MAX_BATCH = BI_ATTN_MAX_BATCH;

template <int D>
struct PCfg {
    static constexpr int NST = D == 64 ? 8 : 4;          // page stages in the ring
    static constexpr int BOXES = D / 64;                 // 64-element (128 B) column boxes
    static constexpr int BOX_BYTES = PAGE * 128;         // one box of a page: 64 rows x 128 B
    static constexpr int PAGE_BYTES = BOXES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;   // K page + V page
    static constexpr int QBOX_BYTES = P_ROWS * 128;
    static constexpr int Q_BYTES = BOXES * QBOX_BYTES;
    static constexpr int RING_OFF = Q_BYTES;             // (P lives in tensor memory)
    static constexpr int BAR_OFF = RING_OFF + NST * STAGE_BYTES;
    // ring (2 NST), s / o full and empty pairs, p full / empty per P buffer, the xs pair,
    // q_full, q_free, and one drain per issuer
    static constexpr int NBARS = 2 * NST + 4 + 2 * P_NPB + 4 + 2 + 4;
    // the barriers, then the tensor-memory address slot (8 bytes), then the (m, l) rows
    static constexpr int XS_OFF = (BAR_OFF + NBARS * 8 + 8 + 15) / 16 * 16;
    static constexpr int XS_BYTES = 2 * P_ROWS * 8;       // per O buffer: (m, l) per row
    static constexpr int MISC_OFF = XS_OFF + XS_BYTES;
    static constexpr int MISC_BYTES = ((P_MAX_BATCH + 1) + 3 * P_MAX_BATCH + 4) * 4;
    // per epilogue warp: 32 O rows of 32 floats, staged for coalesced stores (rows padded
    // to 144 bytes: conflict-free both ways)
    static constexpr int EPI_STRIDE = 32 * 4 + 16;
    static constexpr int EPI_OFF = (MISC_OFF + MISC_BYTES + 15) / 16 * 16;
    static constexpr size_t SMEM = 1024 + size_t(EPI_OFF) + size_t(4 * 32 * EPI_STRIDE);
    static constexpr int S_COL = 0;                       // S buffers: columns [0,64), [64,128)
    static constexpr int O_COL = 2 * PAGE;                // O buffers (by item): D columns each
    // P buffers (by page): 128 rows x 64 keys of bf16, two keys per 32-bit column
    static constexpr int P_TCOL = O_COL + 2 * D;
    static_assert(P_TCOL + P_NPB * (PAGE / 2) <= P_TMEM_COLS, "tensor memory columns");
    static_assert(RING_OFF % 1024 == 0 && BAR_OFF % 1024 == 0, "1024-byte aligned buffers");
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

template <int D>
__global__ void __launch_bounds__(P_THREADS, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_q,
                    const int32_t* __restrict__ block_table, int max_pages, int num_pages,
                    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q,
                    int B, int total_q, int max_q, int max_seq_len, int Hq, int Hkv,
                    float scale_log2, float* __restrict__ ws_o, float* __restrict__ ws_ml,
                    int maxC, unsigned int* err) {
    using C = PCfg<D>;
    constexpr int NST = C::NST;
    constexpr int chunk_pages = CHUNK / PAGE;
    static_assert(chunk_pages <= 32, "an item's block-table entries are read one per lane");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sStage = smem + C::RING_OFF;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + NST;
    uint64_t* s_full = empty + NST;    // scores of page g in S buffer g&1
    uint64_t* s_empty = s_full + 2;    // ... read by the four softmax warps
    uint64_t* p_full = s_empty + 2;    // P of page g in P buffer g%4 (four softmax warps)
    uint64_t* p_empty = p_full + P_NPB;  // P V of page g has completed (MMA commit)
    uint64_t* o_full = p_empty + P_NPB;  // item k's O (buffer k&1) is complete (MMA commit)
    uint64_t* o_empty = o_full + 2;    // ... and read out by the four epilogue warps
    uint64_t* xs_bar = o_empty + 2;    // item k's (m, l) per row are in xs[k&1]
    uint64_t* q_full = xs_bar + 2;     // the Q tile has landed (TMA)
    uint64_t* q_free = q_full + 1;     // every MMA reading the previous Q tile is done
    uint64_t* drain = q_free + 1;      // [2]: S issuer, P V issuer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
    static_assert(C::XS_OFF >= C::BAR_OFF + (2 * NST + 4 + 2 * P_NPB + 4 + 2 + 4) * 8 + 8,
                  "barriers overlap xs");
    float2* xs = reinterpret_cast<float2*>(smem + C::XS_OFF);  // [2][P_ROWS]
    int* prefix = reinterpret_cast<int*>(smem + C::MISC_OFF);  // [B+1] items before sequence b
    int* seq_len = prefix + P_MAX_BATCH + 1;    // per sequence: length, first token, width
    int* seq_t0 = seq_len + P_MAX_BATCH;
    int* seq_qb = seq_t0 + P_MAX_BATCH;
    volatile int* abort_flag = seq_qb + P_MAX_BATCH;
    const unsigned long long wait_ns = wait_budget_ns(err);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv;        // query heads per KV head (divides P_ROWS)
    const int TQ = P_ROWS / G;     // tokens per query tile

    if (warp == P_MMA) {
        tmem_alloc(tmem_slot, P_TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);   // released by the P V warp's commit after P V
        }
        for (int i = 0; i < P_NPB; ++i) {
            mbar_init(&p_full[i], P_NSM);
            mbar_init(&p_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], P_NSM);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 4);
            mbar_init(&xs_bar[i], P_NSM);
        }
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // chunks a query tile reduces: through the chunk of its last token's position
    auto tile_chunks = [&](int L, int qb, int qt) {
        const int last = min(qb, (qt + 1) * TQ) - 1;
        return ((L - qb + last) >> CHUNK_LOG2) + 1;
    };
    // work items per sequence: sum over its query tiles of chunks x KV heads
    for (int b = tid; b < B; b += P_THREADS) {
        const SeqInfo si = seq_info(seq_lens, cu_q, b);
        const bool ok = seq_ok(si, max_q, max_seq_len, total_q);
        if (!ok) latch_error(err, kErrDeviceArg);
        int n = 0;
        if (ok) {
            const int nqt = (si.qb + TQ - 1) / TQ;
            for (int qt = 0; qt < nqt; ++qt) n += tile_chunks(si.L, si.qb, qt);
        }
        prefix[b + 1] = n * Hkv;
        seq_len[b] = si.L;
        seq_t0[b] = si.t0;
        seq_qb[b] = ok ? si.qb : 0;
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
    // this CTA's contiguous run of items (runs differ in length by at most one)
    const int w_begin = int(int64_t(blockIdx.x) * total / gridDim.x);
    const int w_end = int(int64_t(blockIdx.x + 1) * total / gridDim.x);

    // Item cursor (every warp walks the same run): sequence b, query tile qt, KV head h,
    // chunk c (fastest), and the tile's chunk count nch.
    struct Cursor {
        int b, qt, h, c, nch;
    };
    auto seek = [&](int w) {
        Cursor k{B, 0, 0, 0, 1};
        if (w >= total) return k;  // an empty run
        // sequence b with prefix[b] <= w < prefix[b+1]: a valid one (it has items), so
        // its tiles' chunk counts are >= 1 and the walk below ends inside its tiles
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= w) lo = mid; else hi = mid;
        }
        k.b = lo;
        int r = w - prefix[k.b];
        k.qt = 0;
        const int nqt = (seq_qb[k.b] + TQ - 1) / TQ;
        for (;;) {
            k.nch = tile_chunks(seq_len[k.b], seq_qb[k.b], k.qt);
            if (r < k.nch * Hkv || k.qt + 1 >= nqt) break;
            r -= k.nch * Hkv;
            ++k.qt;
        }
        k.h = r / k.nch;
        k.c = r - k.h * k.nch;
        return k;
    };
    auto advance = [&](Cursor& k) {
        if (++k.c < k.nch) return;
        k.c = 0;
        if (++k.h < Hkv) return;
        k.h = 0;
        if (++k.qt * TQ >= seq_qb[k.b]) {
            k.qt = 0;
            do {
                ++k.b;
            } while (k.b < B && prefix[k.b + 1] == prefix[k.b]);
        }
        if (k.b < B) k.nch = tile_chunks(seq_len[k.b], seq_qb[k.b], k.qt);
    };
    // pages of chunk c: those the decode kernel reduces for the chunk, up to the
    // sequence's end (pages past a row's position are masked for it and add +0 to its O
    // and sums; processing the same pages keeps even the signs of zeros identical)
    auto item_pages = [&](const Cursor& k) {
        return min(chunk_pages, (seq_len[k.b] - k.c * CHUNK + PAGE - 1) / PAGE);
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

    if (warp == P_PRODUCER) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        uint32_t g = 0;
        Cursor k = seek(w_begin);
        for (int w = w_begin; ok && w < w_end; ++w, advance(k)) {
            const int npages = item_pages(k);  // <= chunk_pages = 8
            // the item's block-table entries, one per lane, read before the first wait for
            // a free stage: no dependent global load between a stage freeing and its copy
            const int pidx_l = k.c * chunk_pages + lane;
            const int phys_l = (lane < npages && pidx_l < max_pages)
                                   ? block_table[int64_t(k.b) * max_pages + pidx_l]
                                   : -1;
            for (int i = 0; i < npages; ++i, ++g) {
                const int s = int(g % NST);
                if (!wait(&empty[s], ((g / NST) & 1u) ^ 1u)) break;
                const int phys = __shfl_sync(0xffffffffu, phys_l, i);
                if (elect_one()) {
                    const bool valid = phys >= 0 && phys < num_pages;
                    if (valid) {
                        uint8_t* st = sStage + s * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                        const int row = (phys * Hkv + k.h) * PAGE;
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
            if (lane == 0) give_up();
            for (int kk = 1; kk <= NST && kk <= int(g); ++kk) {  // issued copies land (bounded)
                const uint32_t gg = g - kk;
                mbar_wait(&full[gg % NST], (gg / NST) & 1u, nullptr, 100000000ull);
            }
        }
    } else if (warp == P_MMA) {
        // ----------------------------------------------------------------- S issuer
        // S(page) = Q K^T into S buffer (page & 1), as soon as the page has landed and the
        // softmax has read the buffer's previous scores.  At each new Q tile: the S MMAs
        // that read the old tile (the only readers of Q) complete, then this warp copies
        // the new one.
        constexpr uint32_t idesc_s = umma_idesc_bf16(128, PAGE, 0, 0);  // K K-major
        const uint64_t q_desc0 = umma_smem_desc(smem_addr(sQ), 16, 1024, 2);
        const uint64_t k_desc0 = umma_smem_desc(smem_addr(sStage), 16, 1024, 2);
        if (lane == 0) tma_prefetch_desc(&tmap_q);
        uint32_t g = 0, qgen = 0;
        bool q_in_flight = false;
        Cursor k = seek(w_begin);
        for (int w = w_begin; ok && w < w_end; ++w, advance(k)) {
            const int npages = item_pages(k);
            if (w == w_begin || k.c == 0) {
                // a new Q tile: rows r = token (r / G) of the tile x head r mod G
                if (qgen > 0) {
                    if (elect_one()) tc_commit(q_free);
                    __syncwarp();
                    if (!wait(q_free, (qgen - 1u) & 1u)) break;
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(q_full, C::Q_BYTES);
                    const int t0 = seq_t0[k.b] + k.qt * TQ;
#pragma unroll
                    for (int bx = 0; bx < C::BOXES; ++bx)
                        tma_load_3d_s(smem_addr(sQ + bx * C::QBOX_BYTES), &tmap_q, smem_addr(q_full),
                                      bx * 64, k.h * G, t0);
                }
                __syncwarp();
                q_in_flight = true;
                if (!wait(q_full, qgen & 1u)) break;
                q_in_flight = false;
                ++qgen;
            }
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
                        for (int kk = 0; kk < 4; ++kk)         // in 16-wide steps: +32 B
                            tc_mma_bf16(d, q_desc0 + uint64_t(bx * (C::QBOX_BYTES >> 4) + kk * 2),
                                        k_desc + uint64_t(bx * (C::BOX_BYTES >> 4) + kk * 2),
                                        idesc_s, (bx | kk) != 0 ? 1u : 0u);
                    tc_commit(&s_full[sb]);
                }
                __syncwarp();
            }
            g += uint32_t(npages);
        }
        if (!ok) {
            if (lane == 0) give_up();
            // a Q copy still in flight lands before the CTA exits (bounded)
            if (q_in_flight) mbar_wait(q_full, qgen & 1u, nullptr, 100000000ull);
        }
        // every MMA this warp issued completes before tensor memory is released
        if (elect_one()) tc_commit(&drain[0]);
        __syncwarp();
        mbar_wait(&drain[0], 0, nullptr, 100000000ull);
    } else if (warp == P_PV) {
        // --------------------------------------------------------------- P V issuer
        // O(item) += P V of each page once the softmax has written its P (buffer page % 4).
        // The page's S completed before the softmax read it, so this warp's commit after
        // P V marks the whole stage free.
        constexpr uint32_t idesc_pv = umma_idesc_bf16(128, D, 0, 1);    // V N-major
        const uint64_t v_desc0 =
            umma_smem_desc(smem_addr(sStage + C::PAGE_BYTES), C::BOX_BYTES, 1024, 2);
        uint32_t g = 0;
        int item = 0;
        Cursor k = seek(w_begin);
        for (int w = w_begin; ok && w < w_end; ++w, advance(k), ++item) {
            const int npages = item_pages(k);
            const int ob = item & 1;
            for (int i = 0; i < npages; ++i) {
                const uint32_t gi = g + uint32_t(i);
                const int s = int(gi % NST), pb = int(gi % P_NPB);
                if (!wait(&p_full[pb], (gi / P_NPB) & 1u)) break;
                // the O buffer of this item was read out for item-2
                if (i == 0 && !wait(&o_empty[ob], (uint32_t(item >> 1) & 1u) ^ 1u)) break;
                tc_fence_after_sync();
                if (elect_one()) {
                    const uint32_t p_tmem = tmem_base + uint32_t(C::P_TCOL + pb * (PAGE / 2));
                    const uint64_t v_desc = v_desc0 + uint64_t((s * C::STAGE_BYTES) >> 4);
                    const uint32_t o_tmem = tmem_base + uint32_t(C::O_COL + ob * D);
#pragma unroll
                    for (int kk = 0; kk < PAGE / 16; ++kk)  // keys 16kk..: +8 columns of P, +2 KB in V
                        tc_mma_bf16_ts(o_tmem, p_tmem + uint32_t(kk * 8), v_desc + uint64_t(kk * 128),
                                       idesc_pv, (i == 0 && kk == 0) ? 0u : 1u);
                    tc_commit(&p_empty[pb]);
                    tc_commit(&empty[s]);   // K and V of the page are no longer read
                    if (i == npages - 1) tc_commit(&o_full[ob]);
                }
                __syncwarp();
            }
            g += uint32_t(npages);
        }
        if (!ok && lane == 0) give_up();
        if (elect_one()) tc_commit(&drain[1]);
        __syncwarp();
        mbar_wait(&drain[1], 0, nullptr, 100000000ull);
    } else if (warp >= P_EPI) {
        // ------------------------------------------------------------------ epilogue
        // Quarter e = warp mod 4: rows 32e..32e+31 of item k's O (buffer k&1), written
        // with their (m, l) as the chunk partial of every row that reduces the chunk.
        const int e = warp & 3;
        const int r = 32 * e + lane;
        uint8_t* epi_stage = smem + C::EPI_OFF + e * (32 * C::EPI_STRIDE);
        int item = 0;
        Cursor k = seek(w_begin);
        for (int w = w_begin; ok && w < w_end; ++w, advance(k), ++item) {
            const int L = seq_len[k.b], qb = seq_qb[k.b];
            const int j = k.qt * TQ + r / G, gg = r - (r / G) * G;
            const int pos = j < qb ? L - qb + j : -1;
            const int ob = item & 1;
            const uint32_t par = uint32_t(item >> 1) & 1u;
            if (!wait(&xs_bar[ob], par) || !wait(&o_full[ob], par)) break;
            tc_fence_after_sync();
            const float2 ml = xs[ob * P_ROWS + r];
            const bool store = pos >= k.c * CHUNK;
            const int64_t idx =
                (int64_t(seq_t0[k.b] + j) * Hq + int64_t(k.h) * G + gg) * maxC + k.c;
            const uint32_t lane_base = uint32_t(32 * e) << 16;
            // O rows 32 columns at a time, staged through shared memory so that each store
            // instruction writes four rows' 128-byte segments instead of 32 scattered
            // 16-byte pieces
            const int rr = lane >> 3, part = lane & 7;  // reader: row within 4, 16-B piece
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t v[32];
                tmem_load_32x32b_x32_sync(
                    tmem_base + lane_base + uint32_t(C::O_COL + ob * D + cc * 32), v);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    *reinterpret_cast<uint4*>(epi_stage + lane * C::EPI_STRIDE + q4 * 16) =
                        make_uint4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                __syncwarp();
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const int row = 4 * q8 + rr;
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
            if (store) *reinterpret_cast<float2*>(ws_ml + idx * 2) = ml;
        }
        if (!ok && lane == 0) give_up();
    } else {
        // ------------------------------------------------------------------- softmax
        // Warp sw reads tensor-memory lanes 32sw .. 32sw+31: query rows 32sw + lane, all 64
        // keys of every page.
        const int sw = warp;
        const int r = 32 * sw + lane;
        const uint32_t lane_base = uint32_t(32 * sw) << 16;
        uint32_t g = 0;
        int item = 0;
        Cursor k = seek(w_begin);
        for (int w = w_begin; ok && w < w_end; ++w, advance(k), ++item) {
            const int L = seq_len[k.b], qb = seq_qb[k.b];
            const int npages = item_pages(k);
            const int j = k.qt * TQ + r / G;
            const int pos = j < qb ? L - qb + j : -1;
            const int ob = item & 1;
            // whether each page of the item is in the cache, from the block table (the
            // producer's test on the same entries), one page per lane: the softmax needs
            // no stage's landing for it, only for the pages whose V rows it zeroes
            const int pidx_l = k.c * chunk_pages + lane;
            const int phys_l = (lane < npages && pidx_l < max_pages)
                                   ? block_table[int64_t(k.b) * max_pages + pidx_l]
                                   : -1;
            const bool valid_l = phys_l >= 0 && phys_l < num_pages;
            float m_ref = -INFINITY;
            float l_run[4] = {0.f, 0.f, 0.f, 0.f};  // running sums of the four 16-key slices
            for (int i = 0; i < npages && ok; ++i) {
                const uint32_t gi = g + uint32_t(i);
                const int s = int(gi % NST), sb = int(gi & 1u);
                const uint32_t par = (gi >> 1) & 1u;
                const int page0 = k.c * CHUNK + i * PAGE;
                if (!wait(&s_full[sb], par)) break;
                tc_fence_after_sync();
                uint32_t sv[PAGE];
                tmem_load_32x32b_x64_sync(tmem_base + lane_base + uint32_t(C::S_COL + sb * PAGE),
                                          sv);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                const bool valid = __shfl_sync(0xffffffffu, valid_l ? 1 : 0, i) != 0;
                float sl[PAGE];
                if (__all_sync(0xffffffffu, valid && page0 + PAGE - 1 <= pos)) {
                    // every key of the page is visible to every row of the warp
#pragma unroll
                    for (int kk = 0; kk < PAGE; ++kk) sl[kk] = __uint_as_float(sv[kk]);
                } else {
#pragma unroll
                    for (int kk = 0; kk < PAGE; ++kk)
                        sl[kk] = (valid && page0 + kk <= pos) ? __uint_as_float(sv[kk]) : -INFINITY;
                }
                // the exact row max of the page (max does not round: any order), by
                // three-input maxima: 31 instructions instead of 63
                float mt[1];
                {
                    float t1[22], t2[8];
#pragma unroll
                    for (int kk = 0; kk < 21; ++kk)
                        t1[kk] = fmax3(sl[3 * kk], sl[3 * kk + 1], sl[3 * kk + 2]);
                    t1[21] = sl[63];
#pragma unroll
                    for (int kk = 0; kk < 7; ++kk)
                        t2[kk] = fmax3(t1[3 * kk], t1[3 * kk + 1], t1[3 * kk + 2]);
                    t2[7] = t1[21];
                    mt[0] = fmax3(fmax3(t2[0], t2[1], t2[2]), fmax3(t2[3], t2[4], t2[5]),
                                  fmaxf(t2[6], t2[7]));
                }
                const float m_page = mt[0] * scale_log2;
                const bool raise = m_page > m_ref + kRescaleLog2 ||
                                   (m_ref == -INFINITY && m_page != -INFINITY);
                const float factor = raise ? ex2(m_ref - m_page) : 1.f;
                if (raise) m_ref = m_page;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) l_run[q4] *= factor;
                const int pb = int(gi % P_NPB);
                if (!wait(&p_empty[pb], ((gi / P_NPB) & 1u) ^ 1u)) break;
                tc_fence_after_sync();  // P V of page gi-4 read this P buffer: now rewritten
                if (i > 0 && __any_sync(0xffffffffu, raise)) {
                    // this quarter's O rows *= factor once P V of page gi-1 has completed
                    const uint32_t gp = gi - 1u;
                    if (!wait(&p_empty[gp % P_NPB], (gp / P_NPB) & 1u)) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t v[32];
                        const uint32_t ta =
                            tmem_base + lane_base + uint32_t(C::O_COL + ob * D + cc * 32);
                        tmem_load_32x32b_x32_sync(ta, v);
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk)
                            v[kk] = __float_as_uint(__uint_as_float(v[kk]) * factor);
                        tmem_store_32x32b_x32_sync(ta, v);
                    }
                    tc_fence_before_sync();
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                uint32_t pk[PAGE / 2];  // row r of P, two keys per word
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {  // 16-key slice q4
                    float pv[16];
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        pv[kk] = ex2(fmaf(sl[16 * q4 + kk], scale_log2, -m_use));
#pragma unroll
                    for (int kk = 0; kk < 16; kk += 2)
                        pk[8 * q4 + kk / 2] = pack_bf16x2(pv[kk], pv[kk + 1]);
#pragma unroll
                    for (int width = 8; width >= 1; width /= 2)
#pragma unroll
                        for (int kk = 0; kk < width; ++kk) pv[kk] = pv[kk] + pv[kk + width];
                    l_run[q4] = l_run[q4] + pv[0];
                }
                // P into this quarter's lanes of the page's P buffer in tensor memory (the
                // P V MMA reads it from there)
                tmem_store_32x32b_x32_sync(
                    tmem_base + lane_base + uint32_t(C::P_TCOL + pb * (PAGE / 2)), pk);
                // V rows of this warp's 16 keys past the sequence end (or of an invalid
                // page) are zeroed so unwritten cache slots cannot inject NaN/Inf via 0 * v
                const int vend = valid ? L - page0 : 0;
                if (vend < (sw + 1) * 16) {
                    // after the stage's copies have landed (an invalid page's stage had none)
                    if (!wait(&full[s], (gi / NST) & 1u)) break;
                    const int r0 = max(vend, sw * 16);
                    uint8_t* vst = sStage + s * C::STAGE_BYTES + C::PAGE_BYTES;
                    const int n16 = ((sw + 1) * 16 - r0) * 8;  // 16-byte pieces per box
                    for (int idx = lane; idx < C::BOXES * n16; idx += 32) {
                        const int bx = idx / n16, rem = idx - bx * n16;
                        *reinterpret_cast<uint4*>(vst + bx * C::BOX_BYTES + r0 * 128 + rem * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();  // the zeroed V rows, read by the MMA
                }
                tc_fence_before_sync();    // the P stores, before the arrival
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
            }
            if (!ok) break;
            g += uint32_t(npages);
            // (m, l) of each row for the epilogue, once it has read this buffer's previous
            // contents (item-2); the slice sums in ascending slice order
            if (!wait(&o_empty[ob], (uint32_t(item >> 1) & 1u) ^ 1u)) break;
            xs[ob * P_ROWS + r] = make_float2(m_ref, ((l_run[0] + l_run[1]) + l_run[2]) + l_run[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&xs_bar[ob]);
        }
        if (!ok && lane == 0) give_up();
    }
    // every warp is done with tensor memory and shared memory past this barrier
    tc_fence_before_sync();
    __syncthreads();
    if (warp == P_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, P_TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_prefill_t(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                             float scale, void* out, float* lse, void* workspace,
                             cudaStream_t stream) {
    using Cf = PCfg<D>;
    const uint64_t rows = uint64_t(a.num_pages) * uint64_t(a.hkv) * PAGE;
    const int G = int(a.hq / a.hkv);
    CUtensorMap tk, tv, tq;
    if (!tmap_2d_bf16(&tk, a.k_cache, D, rows, D, 64, PAGE, 128) ||
        !tmap_2d_bf16(&tv, a.v_cache, D, rows, D, 64, PAGE, 128) ||
        !tmap_3d_bf16(&tq, q, D, uint64_t(a.hq), uint64_t(a.total_q), D, uint64_t(a.hq) * D, 64,
                      uint32_t(G), uint32_t(P_ROWS / G)))
        return cudaErrorNotSupported;
    auto kern = attn_prefill_kernel<D>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(Cf::SMEM));
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    const int maxC = int((a.max_seq_len + CHUNK - 1) / CHUNK);
    // items: at most batch x query tiles x chunks x KV heads
    const int64_t tiles_bound = (a.total_q + P_ROWS / G - 1) / (P_ROWS / G) + a.batch;
    const int64_t items_bound = tiles_bound * int64_t(maxC) * a.hkv;
    if (items_bound > 0x7fffffffLL) return cudaErrorNotSupported;
    const int grid = int(items_bound < dev.num_sms ? items_bound : dev.num_sms);
    float* ws_o = static_cast<float*>(workspace);
    float* ws_ml = ws_o + a.total_q * a.hq * int64_t(maxC) * D;
    cudaError_t e = launch_pdl(kern, dim3(grid), dim3(P_THREADS), Cf::SMEM, stream, tk, tv, tq,
                               a.block_table, int(a.max_pages), int(a.num_pages), a.seq_lens,
                               a.cu_q, int(a.batch), int(a.total_q), int(a.max_q),
                               int(a.max_seq_len), int(a.hq), int(a.hkv), scale * kLog2e, ws_o,
                               ws_ml, maxC, dev.err_word);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(a, workspace, CHUNK_LOG2, out, lse, nullptr, dev.err_word, stream);
}

}  // namespace

cudaError_t launch_prefill(const DeviceInfo& dev, const void* q, const PagedArgs& a,
                           float scale, void* out, float* lse, void* workspace,
                           cudaStream_t stream) {
    return a.head_dim == 64
               ? launch_prefill_t<64>(dev, q, a, scale, out, lse, workspace, stream)
               : launch_prefill_t<128>(dev, q, a, scale, out, lse, workspace, stream);
}

}  // namespace bi
