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
//   * the kind::f16 instruction (tcgen05.mma.cta_group::1, bf16 or binary16 in, fp32
//     accumulator in tensor memory) and its 16-wide K step: each element adds the 16
//     products of one K slice to its own fp32 accumulator;
//   * the K order: 64-wide K-blocks in ascending order, and inside a block the four
//     16-wide steps in ascending order, the first one overwriting the accumulator;
//   * the epilogue: fp32 -> bf16 (or binary16) round-to-nearest-even, or fp32 as is.
// What follows M (scheduling, and the instruction's shape):
//   * the instruction's height: 64 rows when a tile stages at most 64 rows (row 16q+r in
//     tensor-memory lane 32q+r), else 128 (row m in lane m % 128);
//   * the instruction's width, 32 to 256 columns: one instruction covers the CTA tile's
//     nsub 32-column sub-tiles;
//   * the CTA tile, from a cost model (gemm_schedule): 128 x 32*nsub, or 256 x 256 (two
//     instructions along M) for large M, so different M run different template instances;
//   * a_rows: how many X rows are staged per K-block (M rounded up to 8, at most 128, or
//     256); rows past a_rows land in lanes that are never stored;
//   * kbs and stages: how many K-blocks one ring stage carries and how deep the ring is.
// The book chapter's Case 6 names a smaller instruction at small M as one way to break
// invariance, because an instruction may group or round its products differently.  Here
// the shape changes, so the invariance rests on each element's 16-product step not
// depending on the instruction's height or width.  That is a property of the hardware,
// not of this code; the tests pin it on fp32 accumulator bits with operands built to
// expose any regrouping (cancelling pairs of large products, subnormal inputs and
// products) at every height and width the schedule picks, both layouts, bf16, binary16
// and quantized W.
//
// Warp roles (192 threads, persistent, one CTA per SM): warp 0 = TMA producer, warp 1 =
// TMEM allocator + MMA issuer, warps 2..5 = epilogue (tcgen05.ld -> convert -> global).
// Producer and MMA warps run their loops with all 32 lanes converged and let one
// elected lane issue each TMA / tcgen05 instruction.  Full/empty mbarriers guard the
// ring; two TMEM accumulators let the epilogue of tile i overlap the main loop of tile
// i+1.  Descriptors and shared addresses are computed once and advanced by adds in the
// issue loops (per-instruction descriptor arithmetic was measured to double the cost of
// each MMA).  W layout NK ([N,K]) feeds the MMA as a K-major operand with 128-byte
// swizzle, layout KN ([K,N]) as an N-major operand with 128-byte swizzle.  When K is a
// multiple of 64 one rank-3 TMA copy per operand brings all the K-blocks of a stage.
// Every mbarrier wait is bounded: a wait that runs out latches the device error word,
// raises a CTA-wide abort flag, drains outstanding copies and MMAs (bounded), frees
// tensor memory and returns.
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace bi {
namespace {

#ifndef BI_GEMM_BN
#define BI_GEMM_BN 32
#endif

constexpr int BM = 128;                     // rows of an M-tile (64-row instructions below 65)
constexpr int BN = BI_GEMM_BN;              // columns of a sub-tile (an instruction spans nsub)
constexpr int BK = 64;                      // K-block: one 128-byte swizzle row of bf16
constexpr int UK = 16;                      // K of one kind::f16 instruction
constexpr int MAX_NSUB = 256 / BN;          // two accumulators of nsub*BN columns in 512
constexpr int MAX_KBS = 8;                  // K-blocks per ring stage (K-major operands)
constexpr int MAX_KBS_KN = 4;               // N-major W: one box spans 64*kbs <= 256 k-rows
constexpr int MAX_STAGES = 48;
constexpr int MAX_SPLITS = 8;               // split-K cluster size (portable maximum)
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
// Quantized W: eight (or sixteen, see conv_warps) more warps from warp 6 on turn the
// packed codes of each stage into bf16 operand tiles.  The ring (at most MAX_QSTAGES
// stages) holds X blocks and packed codes only; the bf16 tiles live in a separate ring of
// MAX_QWBUF buffers.
constexpr int CONV_WARPS = 8;
// Converter warps of a QUANT kernel: sixteen (two groups of eight, each group's two halves
// taking alternate K-blocks of a stage) for transposed-layout W in 32-column tiles (small
// M: the conversion sets the pace and the registers allow 704 threads), else eight.
__host__ __device__ constexpr int conv_warps(bool kn, int nsub) {
    return !kn && nsub == 1 ? 2 * CONV_WARPS : CONV_WARPS;
}
__host__ __device__ constexpr int gemm_threads(bool quant, bool kn, int nsub) {
    return quant ? THREADS + 32 * conv_warps(kn, nsub) : THREADS;
}
constexpr int MAX_QSTAGES = 16;
constexpr int MAX_QWBUF = 4;
constexpr int Q_SROW = 16;     // bytes of staged scales (or biases) per tile row, one K-block
constexpr int Q_SROW_KBS = 64; // ... for stages of several K-blocks (up to 8)
constexpr int B_KB_BYTES = BN * BK * 2;     // one instruction tile's W block per K-block
constexpr int A_MMA_BYTES = BM * BK * 2;    // 16 KiB: what one MMA reads from an X block
constexpr int SMEM_BYTES = 220 * 1024;      // dynamic shared memory per CTA
constexpr int CTRL_BYTES = 1024;            // barriers and flags at the end
constexpr int RING_BYTES = SMEM_BYTES - 1024 /* alignment slack */ - CTRL_BYTES;
// N-major W (layout KN): one swizzle atom spans min(BN, 64) columns
constexpr int KN_ATOM_N = BN < 64 ? BN : 64;
constexpr int KN_ATOM_BYTES = KN_ATOM_N * 2 * BK;  // one atom column of a K-block
constexpr int KN_SWIZZLE = KN_ATOM_N * 2;          // 64 or 128 bytes
// Dense W in layout KN can be staged in atoms of 64 columns (128-byte rows, 128-byte
// swizzle), so that every TMA row segment is a whole 128-byte line: always for tiles of 64
// columns or more, and for 32-column tiles when few X rows are staged (the W stream sets
// the pace there; a 32-column tile then stages the 64-column atom that holds it, twice its
// own bytes from L2, and its MMA starts 64 bytes into each row).  Otherwise, and for
// quantized natural-layout W (whose converters write KN_ATOM_N atoms), KN_ATOM_N atoms.
constexpr int DKN_ATOM_N = 64;
constexpr int DKN_MAX_ROWS = 32;  // X rows staged at most for the wide atoms of 32-column tiles
__host__ __device__ constexpr int dkn_cols(int nsub) {  // W columns staged per K-block
    return nsub * BN > DKN_ATOM_N ? nsub * BN : DKN_ATOM_N;
}
// Quantized W in the natural layout: K-blocks per stage for a tile of nsub instruction
// tiles, so that a converter thread holds at most 8 prefetched scale codes (its pieces
// per K-block: nsub*BN/16) and a code box spans at most 256 k-rows
__host__ __device__ constexpr int qkn_max_kbs(int nsub) {
    return nsub * BN / 16 >= 8 ? 1 : (8 / (nsub * BN / 16) < MAX_KBS_KN ? 8 / (nsub * BN / 16)
                                                                        : MAX_KBS_KN);
}

static_assert(BN == 32 || BN == 64, "instruction sub-tile N must be 32 or 64");
static_assert((2 * MAX_STAGES + 7 + 2 * MAX_QWBUF) * 8 + 16 <= CTRL_BYTES,
              "control block too small");

struct GemmArgs {
    void* y;
    int64_t ldy;
    int M, N, K;
    int a_rows;          // X rows staged per K-block (multiple of 8, <= 128)
    int nsub;            // instruction tiles per CTA tile along N
    int kbs;             // K-blocks per ring stage
    int blocked;         // K % 64 == 0: one rank-3 copy per operand per stage
    int stages;          // ring depth
    int w_stream_once;   // one M-tile: W is read exactly once (L2 evict-first hint)
    int w_early;         // W (codes, scales, biases) may be read before the previous grid
                         // in the stream has finished: the caller has promised that grid
                         // does not write them
    // Split-K (the non-invariant kernel only): a cluster of `splits` CTAs shares each
    // output tile, CTA rank r accumulating K-blocks [r*kb_per_split, (r+1)*kb_per_split).
    // The invariant kernel has splits = 1 and kb_per_split = the number of K-blocks.
    int splits;
    int kb_per_split;
    int f16;           // X, W (and a 16-bit Y) are IEEE binary16 instead of bf16
    // Quantized W (QUANT kernels only): format (0 mxfp4, 1 nvfp4, 2 mxfp8, 3 affine 4-bit,
    // 4 affine 8-bit), group size, per-group scales (bytes, or bf16 for affine, row
    // stride lds) and affine biases (bf16, row stride ldb); packed bytes per row per K-block.
    int qfmt;
    int gs;
    const void* qscales;
    int64_t lds;
    const uint16_t* qbiases;
    int64_t ldb;
    int q_kb_bytes;
    int wbufs;         // bf16 W tile buffers (even, <= MAX_QWBUF)
    int q_staged;      // the scales (and biases) come with the codes, by TMA, q_srow bytes
                       // per row and stage starting at a 16-byte boundary; else the
                       // converters load them from global memory (then kbs = 1)
    int q_srow;        // Q_SROW (one K-block per stage) or Q_SROW_KBS
    int kn_wide;       // dense layout-KN W staged in 64-column atoms (see DKN_ATOM_N)
};

// ----------------------------------------------------------- quantized-code decoding
// From the format definitions (OCP Microscaling FP8 E4M3 and E8M0 scale codes; FP8 E4M3
// elements go through the hardware's exact two-at-a-time conversion below, FP4 E2M1
// elements through a byte lookup); every decoded value is exact in fp32 and in bf16.
__device__ __forceinline__ float dec_e4m3(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float mag;
    if (e == 15u && m == 7u) mag = __uint_as_float(0x7fc00000u);
    else if (e == 0u) mag = float(m) * 0.001953125f;  // m * 2^-9
    else mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (c & 0x80u) ? -mag : mag;
}

// Two codes to two halves, exactly (every FP8 E4M3 value is a binary16 value): the low
// byte to the low half.
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two) {
    uint32_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(d) : "r"(two));
    return d;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h2) {
    return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

__device__ __forceinline__ float dec_e8m0(uint32_t c) {
    return c == 255u ? __uint_as_float(0x7fc00000u)
                     : (c == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(c << 23));
}

// Byte permute (PTX prmt, default mode): byte n of the result is byte (sel nibble n & 7)
// of the pair {b, a} (a = bytes 0-3); a nibble with bit 3 set instead fills the byte
// with copies of the selected byte's top bit.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Eight FP4 E2M1 codes (one word, low nibble first) to four bf16x2 words, exactly and
// without conversion instructions: the bf16 of each magnitude (0, 0.5, 1, 1.5, 2, 3, 4,
// 6) is looked up one byte at a time, and each code's sign bit becomes its half's.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t (&o)[4]) {
    // low bytes of the eight magnitudes: 00 00 80 c0 00 40 80 c0; high: 00 3f 3f 3f 40 40 40 40
    constexpr uint32_t LO_A = 0xc0800000u, LO_B = 0xc0804000u;
    constexpr uint32_t HI_A = 0x3f3f3f00u, HI_B = 0x40404040u;
    const uint32_t m = w & 0x77777777u;  // one magnitude index per nibble
    const uint32_t lo03 = prmt(LO_A, LO_B, m), hi03 = prmt(HI_A, HI_B, m);
    const uint32_t lo47 = prmt(LO_A, LO_B, m >> 16), hi47 = prmt(HI_A, HI_B, m >> 16);
    // code 2j+1's sign is the top bit of byte j of w, code 2j's that of byte j of w << 4
    const uint32_t w4 = w << 4;
    o[0] = prmt(lo03, hi03, 0x5140u) | (prmt(w, w4, 0x80c0u) & 0x80008000u);
    o[1] = prmt(lo03, hi03, 0x7362u) | (prmt(w, w4, 0x90d0u) & 0x80008000u);
    o[2] = prmt(lo47, hi47, 0x5140u) | (prmt(w, w4, 0xa0e0u) & 0x80008000u);
    o[3] = prmt(lo47, hi47, 0x7362u) | (prmt(w, w4, 0xb0f0u) & 0x80008000u);
}

// An integer code c < 2^23 as fp32 without a conversion instruction: the bits of 2^23 + c
// (byte `byte_sel` of `word` placed in the mantissa's low byte) minus 2^23, exact.
__device__ __forceinline__ float byte_to_f32(uint32_t word, uint32_t byte_sel) {
    return __uint_as_float(prmt(word, 0x4b000000u, 0x7440u | byte_sel)) - 8388608.0f;
}

template <bool KN, bool F32OUT, int NSUB, bool SPLIT, int MSUB, bool QUANT>
__global__ void __launch_bounds__(gemm_threads(QUANT, KN, NSUB), 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_b,
            const GemmArgs args, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int S = args.stages;
    constexpr int nsub = NSUB;
    const int kbs = args.kbs;
    const int a_bytes = args.a_rows * (BK * 2);   // one X block (one K-block)
    // one W block (one K-block, every sub-tile; wide KN atoms: whole 64-column atoms)
    const bool DKN = KN && !QUANT && args.kn_wide != 0;
    const int WA_N = DKN ? DKN_ATOM_N : KN_ATOM_N;            // N-major atom columns
    const int WA_BYTES = WA_N * 2 * BK;                       // one atom of a K-block
    const int WA_SW = WA_N * 2;                               // its swizzle (bytes)
    const uint32_t WA_LAYOUT = WA_SW == 128 ? 2u : 4u;
    const int b_bytes = DKN ? dkn_cols(NSUB) * BK * 2 : nsub * B_KB_BYTES;
    uint8_t* sA = smem;                           // S*kbs X blocks
    uint8_t* sB = smem + S * kbs * a_bytes;       // S*kbs W blocks (QUANT: wbufs W tiles)
    uint8_t* sR = sB + (QUANT ? args.wbufs : S) * kbs * b_bytes;  // QUANT: S code blocks
    // QUANT stage: the packed codes, then (staged) a block of scales and, affine, biases
    const bool q_aff = args.qfmt >= 3;
    const int codes_bytes = nsub * BN * args.q_kb_bytes * kbs;  // rows of kbs K-blocks
    const int s_row = args.q_srow;
    const int s_blk = nsub * BN * s_row;
    const int r_bytes = codes_bytes + (args.q_staged ? (q_aff ? 2 : 1) * s_blk : 0);
    const int gsh = QUANT ? 31 - __clz(args.gs) : 0;  // the group size is a power of two
    const int s_epb = q_aff ? Q_SROW / 2 : Q_SROW;     // window alignment (16 bytes), elements
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
    uint64_t* empty = full + MAX_STAGES;
    uint64_t* tfull = empty + MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* red_full = drain + 1;  // split-K, rank 0: the other ranks' partials are in
    uint64_t* red_free = drain + 2;  // split-K, rank > 0: rank 0 has read this rank's slot
    uint64_t* conv = drain + 3;             // QUANT: W tile buffer b is written
    uint64_t* wfree = conv + MAX_QWBUF;     // QUANT: the MMAs reading buffer b are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wfree + MAX_QWBUF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const unsigned long long wait_ns = wait_budget_ns(err);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N, K = args.K;
    const int tile_n = nsub * BN;
    constexpr int TILE_M = BM * MSUB;             // rows per CTA tile: MSUB instruction tiles
    const int m_tiles = (M + TILE_M - 1) / TILE_M;
    const int n_tiles = (N + tile_n - 1) / tile_n;
    const int num_tiles = m_tiles * n_tiles;
    const int nkb = (K + BK - 1) / BK;
    // Tiles are dealt out to CTAs (to clusters of `splits` CTAs when split), and this CTA
    // accumulates K-blocks [kb0, kb1) of each of its tiles.
    int rank = 0, first_tile = int(blockIdx.x), tile_step = int(gridDim.x);
    if constexpr (SPLIT) {
        rank = int(cluster_ctarank());
        first_tile = int(cluster_id_x());
        tile_step = int(cluster_count_x());
    }
    const int kb0 = rank * args.kb_per_split;
    const int kb1 = kb0 + args.kb_per_split < nkb ? kb0 + args.kb_per_split : nkb;
    // two accumulators (the epilogue of one tile overlaps the next tile's main loop) when
    // they fit in the 512 tensor-memory columns, else one
    constexpr int NACC = 2 * MSUB * NSUB * BN <= 512 ? 2 : 1;
    constexpr int ACC_COLS = MSUB * NSUB * BN;
    const uint32_t tmem_cols = uint32_t(NACC * ACC_COLS);  // a power of two

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        if (QUANT) {
            for (int b = 0; b < args.wbufs; ++b) {
                mbar_init(&conv[b], conv_warps(KN, NSUB) / 2);  // the warps of a group
                mbar_init(&wfree[b], 1);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], EPI_THREADS);
        }
        mbar_init(drain, 1);
        if constexpr (SPLIT) {
            mbar_init(red_full, uint32_t((args.splits - 1) * EPI_THREADS));
            mbar_init(red_free, EPI_THREADS);
        }
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
    // the other CTAs of the cluster signal this CTA's barriers: all are initialised first
    if constexpr (SPLIT) cluster_sync_all();
    const uint32_t tmem_base = *tmem_slot;
    // The set-up above touches no global memory.  The previous grid in the stream may
    // still be running: the producer (and the converters) read W before waiting for that
    // grid only when the caller has allowed it (w_early), X always after; the epilogue
    // waits before its first store; the MMA warp touches only shared and tensor memory.
    pdl_trigger();

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
        const uint32_t sA_s = smem_addr(sA), sB_s = smem_addr(sB), full_s = smem_addr(full);
        const uint32_t stage_a = uint32_t(kbs * a_bytes), stage_b = uint32_t(kbs * b_bytes);
        const bool w_once = args.w_stream_once != 0;
        const bool blocked = args.blocked != 0;
        // W blocks of K-blocks kb .. kb+kbs-1 of tile column n0 into stage `st`
        auto issue_w = [&](uint32_t st, int n0, int kb, int nk) {
            const uint32_t bar = full_s + st * 8u;
            const uint32_t b_dst = sB_s + st * stage_b;
            if (QUANT && KN) {
                // natural layout: the K-block's 64 rows of packed codes, columns n0.. of
                // the tile (x in bytes: n0 * bits / 8)
                // (rows of the stage's kbs K-blocks: one box of 64*kbs rows, zeros past K)
                const uint32_t r_dst = smem_addr(sR) + st * uint32_t(r_bytes);
                const int xb = (n0 * args.q_kb_bytes) / BK;
                if (w_once)
                    tma_load_2d_s_hint(r_dst, &tmap_w, bar, xb, kb * BK, w_policy);
                else
                    tma_load_2d_s(r_dst, &tmap_w, bar, xb, kb * BK);
            } else if (QUANT) {
                // the packed codes of the K-block (one stage = one K-block), rows n0..
                const uint32_t r_dst = smem_addr(sR) + st * uint32_t(r_bytes);
                if (w_once)
                    tma_load_2d_s_hint(r_dst, &tmap_w, bar, kb * args.q_kb_bytes, n0, w_policy);
                else
                    tma_load_2d_s(r_dst, &tmap_w, bar, kb * args.q_kb_bytes, n0);
                if (args.q_staged) {
                    // the groups of the K-block, from the 16-byte boundary at or below
                    // its first group (the block's groups all fall in the 16 bytes)
                    const int xs = ((kb * BK) >> gsh) & ~(s_epb - 1);
                    tma_load_2d_s(r_dst + uint32_t(codes_bytes), &tmap_s, bar, xs, n0);
                    if (q_aff)
                        tma_load_2d_s(r_dst + uint32_t(codes_bytes + s_blk), &tmap_b, bar, xs, n0);
                }
            } else if (KN) {
                // per swizzle atom (WA_N columns) one box of 64*kbs k-rows, from the atom
                // that holds column n0 (a 32-column tile shares its atom with the next
                // tile's CTA: no evict-first hint then, so the line waits in L2 for it)
                const int na = n0 / WA_N * WA_N;
                const int cols = DKN ? dkn_cols(NSUB) : tile_n;
                for (int c = 0; c < cols; c += WA_N) {
                    const uint32_t dst = b_dst + uint32_t(c / WA_N) * uint32_t(kbs * WA_BYTES);
                    if (w_once && cols == tile_n)
                        tma_load_2d_s_hint(dst, &tmap_w, bar, na + c, kb * BK, w_policy);
                    else
                        tma_load_2d_s(dst, &tmap_w, bar, na + c, kb * BK);
                }
            } else if (blocked) {
                if (w_once)
                    tma_load_3d_s_hint(b_dst, &tmap_w, bar, 0, n0, kb, w_policy);
                else
                    tma_load_3d_s(b_dst, &tmap_w, bar, 0, n0, kb);
            } else {
                for (int i = 0; i < nk; ++i) {
                    const uint32_t dst = b_dst + uint32_t(i * b_bytes);
                    if (w_once)
                        tma_load_2d_s_hint(dst, &tmap_w, bar, (kb + i) * BK, n0, w_policy);
                    else
                        tma_load_2d_s(dst, &tmap_w, bar, (kb + i) * BK, n0);
                }
            }
        };
        // X blocks of K-blocks kb .. kb+kbs-1 of tile row m0 into stage `st`
        auto issue_x = [&](uint32_t st, int m0, int kb, int nk) {
            const uint32_t bar = full_s + st * 8u;
            const uint32_t a_dst = sA_s + st * stage_a;
            if (blocked) {
                tma_load_3d_s(a_dst, &tmap_x, bar, 0, m0, kb);
            } else {
                for (int i = 0; i < nk; ++i)
                    tma_load_2d_s(a_dst + uint32_t(i * a_bytes), &tmap_x, bar, (kb + i) * BK, m0);
            }
        };
        // a rank-3 copy always delivers all kbs blocks (zeros past K), a rank-2 copy one
        // block; N-major W boxes always span kbs blocks
        auto stage_tx = [&](int nk) {
            const int x_blocks = blocked ? kbs : nk;
            const int w_blocks = (blocked || KN) ? kbs : nk;
            if (QUANT) return uint32_t(x_blocks * a_bytes + r_bytes);
            return uint32_t(x_blocks * a_bytes + w_blocks * b_bytes);
        };

        // With w_early, before the previous grid is done: W of the first tile's first
        // stages goes straight into the (empty) ring, so the weight stream overlaps the
        // previous kernel's tail.  Without it the wait comes first (the previous grid may
        // have written W) and the same copies are simply the ring's first.
        if (!args.w_early) pdl_wait();
        // At most two stages of W go out before X: the SM's TMA unit serves copies in
        // order, so the first X block would otherwise queue behind the whole ring of W
        const int EARLY_W = S < 2 ? S : 2;
        int early = 0;  // stages of the first tile whose W is already issued
        if (first_tile < num_tiles) {
            const int n0 = (first_tile % n_tiles) * tile_n;
            for (int kb = kb0; kb < kb1 && early < EARLY_W; kb += kbs, ++early) {
                const int nk = kb1 - kb < kbs ? kb1 - kb : kbs;
                if (elect_one()) {
                    mbar_arrive_expect_tx_s(full_s + uint32_t(early) * 8u, stage_tx(nk));
                    issue_w(uint32_t(early), n0, kb, nk);
                }
                __syncwarp();
            }
        }
        pdl_wait();

        for (int t = first_tile; ok && t < num_tiles; t += tile_step) {
            const int mt = t / n_tiles, nt = t % n_tiles;
            const int m0 = mt * TILE_M, n0 = nt * tile_n;
            for (int kb = kb0; kb < kb1; kb += kbs) {
                if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, wait_ns)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const int nk = kb1 - kb < kbs ? kb1 - kb : kbs;  // K-blocks in this stage
                    if (int(issued) >= early) {
                        mbar_arrive_expect_tx_s(full_s + stage * 8u, stage_tx(nk));
                        issue_w(stage, n0, kb, nk);
                    }
                    issue_x(stage, m0, kb, nk);
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
        // One instruction of N = NSUB*BN covers every sub-tile and reads each X block once
        // per k16 step.  K-major W: the tile's rows are contiguous (8-row groups 1024 B
        // apart); N-major W: its swizzle-atom columns sit the descriptor's leading-byte
        // offset apart.
        // A tile of at most 64 rows (M <= 64) runs M = 64 instructions: half the X bytes
        // read per instruction, the same per-element products and K order
        const bool m64 = MSUB == 1 && args.a_rows <= 64;
        const uint32_t idesc =
            umma_idesc_bf16(m64 ? 64 : BM, NSUB * BN, 0, KN ? 1 : 0, args.f16 != 0);
        // X: K-major, 128-byte swizzle, 8-row groups 1024 B apart; +32 B per k16 step
        const uint64_t a_desc0 = umma_smem_desc(smem_addr(sA), 16, 1024, 2);
        // W, layout NK: K-major like X.  Layout KN: N-major; k-rows of WA_SW bytes, 8
        // k-rows per swizzle-atom group, atoms of WA_N columns WA_BYTES apart; a k16 step
        // skips 16 k-rows
        // (KN: a stage holds, per atom of WA_N columns, kbs K-blocks of 64 k-rows, so
        // atoms sit kbs*WA_BYTES apart and K-blocks WA_BYTES apart)
        const uint64_t b_desc0 = KN ? umma_smem_desc(smem_addr(sB), uint32_t(kbs * WA_BYTES),
                                                     8 * WA_SW, WA_LAYOUT)
                                    : umma_smem_desc(smem_addr(sB), 16, 1024, 2);
        constexpr int A_K16 = (UK * 2) >> 4;
        const int B_K16 = KN ? (UK * WA_SW) >> 4 : (UK * 2) >> 4;
        const uint64_t a_step = uint64_t(a_bytes >> 4);
        const uint64_t b_step = uint64_t((KN ? WA_BYTES : b_bytes) >> 4);
        const uint32_t stage_a = uint32_t(kbs * a_bytes), stage_b = uint32_t(kbs * b_bytes);
        const uint32_t empty_s = smem_addr(empty);
        uint32_t stage = 0, phase = 0;
        uint32_t wb = 0, wphase = 0;  // QUANT: the W tile buffer and its phase
        bool ok = true;
        int local = 0;
        for (int t = first_tile; ok && t < num_tiles; t += tile_step, ++local) {
            const int acc = local % NACC;
            const uint32_t acc_phase = uint32_t(local / NACC) & 1u;
            if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, abort_flag, wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + uint32_t(acc * ACC_COLS);
            // dense KN, 32-column tile: its columns start 64 bytes into the atom's rows
            const uint64_t b_col = DKN ? uint64_t((((t % n_tiles) * tile_n) % WA_N) * 2 >> 4) : 0;
            for (int kb = kb0; kb < kb1; kb += kbs) {
                if (!mbar_wait_warp(&full[stage], phase, abort_flag, wait_ns) ||
                    (QUANT && !mbar_wait_warp(&conv[wb], wphase, abort_flag, wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int nk = kb1 - kb < kbs ? kb1 - kb : kbs;
                if (elect_one()) {
                    // descriptors are advanced by adding (byte offset >> 4) to the start-
                    // address field; shared addresses stay below 2^18 so it never carries
                    uint64_t a_blk = a_desc0 + (uint64_t(stage * stage_a) >> 4);
                    uint64_t b_blk = b_desc0 + (uint64_t((QUANT ? wb : stage) * stage_b) >> 4) +
                                     b_col;
                    for (int i = 0; i < nk; ++i, a_blk += a_step, b_blk += b_step) {
                        const uint32_t first = (kb + i) == kb0 ? 1u : 0u;
#pragma unroll
                        for (int k = 0; k < BK / UK; ++k) {
#pragma unroll
                            for (int ms = 0; ms < MSUB; ++ms) {
                                // instruction tile ms: X rows 128ms.., accumulator columns
                                // ms*NSUB*BN..
                                const uint64_t a_desc = a_blk + uint64_t(k * A_K16) +
                                                        uint64_t(ms * (A_MMA_BYTES >> 4));
                                uint64_t b_desc = b_blk + uint64_t(k * B_K16);
                                uint32_t d = d_tmem + uint32_t(ms * NSUB * BN);
                                tc_mma_bf16(d, a_desc, b_desc, idesc, (first && k == 0) ? 0u : 1u);
                            }
                        }
                    }
                    tc_commit_s(empty_s + stage * 8u);  // frees the stage once these MMAs finish
                    if (QUANT) tc_commit(&wfree[wb]);     // and the W tile buffer
                }
                __syncwarp();
                if (++stage == uint32_t(S)) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (QUANT && ++wb == uint32_t(args.wbufs)) {
                    wb = 0;
                    wphase ^= 1u;
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
    } else if (warp < 6) {
        // ------------------------------------------------------------------ epilogue
        pdl_wait();  // Y may still be read by the previous grid
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        // M = 128 instructions: tile row i in lane i.  M = 64 instructions (tiles of at most
        // 64 rows): rows 16q .. 16q+15 in lanes 32q .. 32q+15; the other lanes hold no row
        // (given a row index past the tile, so nothing reads or writes for them)
        const bool m64 = MSUB == 1 && args.a_rows <= 64;
        const int row_in_tile =
            !m64 ? quad * 32 + lane : (lane < 16 ? quad * 16 + lane : BM + lane);
        int local = 0;
        void* const y = args.y;
        const int64_t ldy = args.ldy;
        const bool vec_ok = F32OUT ? ((ldy % 4) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0)
                                   : ((ldy % 8) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0);
        const bool h16 = args.f16 != 0;
        // Split-K: rank r > 0 hands its fp32 partial to rank 0 through rank 0's shared
        // memory (slot r-1 at the top of the ring area: a_rows rows of tile_n floats, the
        // 16-byte pieces of row i rotated by i & 7 so that a warp's stores and loads hit
        // distinct banks); rank 0 adds the slots to its own accumulator in ascending rank
        // order, i.e. in ascending K.  Only warps whose lanes hold staged rows (live) touch
        // tensor memory or the slots; every epilogue thread joins every barrier.
        const int red_rows = args.a_rows;
        const bool live = !SPLIT || quad * (m64 ? 16 : 32) < red_rows;
        const bool red_row = row_in_tile < red_rows;
        const uint32_t slot_bytes = uint32_t(red_rows * tile_n * 4);
        const uint32_t red_base =
            smem_addr(smem + RING_BYTES) - uint32_t(args.splits - 1) * slot_bytes;
        const uint32_t row_off = uint32_t(row_in_tile * tile_n * 4);
        const uint32_t rot = uint32_t(row_in_tile & 7);
        uint32_t to_slot = 0, to_full = 0;
        if (SPLIT && rank != 0) {
            to_slot = cluster_map(red_base + uint32_t(rank - 1) * slot_bytes, 0);
            to_full = cluster_map(smem_addr(red_full), 0);
        }
        for (int t = first_tile; t < num_tiles; t += tile_step, ++local) {
            const int acc = local % NACC;
            const uint32_t acc_phase = uint32_t(local / NACC) & 1u;
            if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, wait_ns)) {
                if (!*abort_flag) fail();
                break;
            }
            if (SPLIT) {
                // rank 0: every partial of this tile has arrived; rank > 0: rank 0 has
                // read this rank's previous partial out of the slot
                const bool got = rank == 0
                    ? mbar_wait_warp<true>(red_full, uint32_t(local & 1), abort_flag, wait_ns)
                    : mbar_wait_warp<true>(red_free, uint32_t(local & 1) ^ 1u, abort_flag, wait_ns);
                if (!got) {
                    if (!*abort_flag) fail();
                    break;
                }
            }
            tc_fence_after_sync();
            const int mt = t / n_tiles, nt = t % n_tiles;
#pragma unroll 1
            for (int ms = 0; ms < MSUB; ++ms)
            for (int c = 0; c < tile_n; c += 32) {
                const int64_t gm = int64_t(mt) * TILE_M + ms * BM + row_in_tile;
                uint32_t r[32];
                if (live) {
                    tmem_load_32x32b_x32(tmem_base + (uint32_t(quad * 32) << 16) +
                                             uint32_t(acc * ACC_COLS + ms * NSUB * BN + c),
                                         r);
                    tmem_load_wait();
                }
                if (SPLIT && rank != 0) {
                    if (live && red_row) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            st_cluster_v4(to_slot + row_off +
                                              ((uint32_t(c / 4 + q) ^ rot) << 4),
                                          r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                    }
                    continue;  // rank > 0 writes nothing to Y
                }
                if (SPLIT && live && red_row) {
                    for (int sp = 1; sp < args.splits; ++sp) {
                        const uint32_t src = red_base + uint32_t(sp - 1) * slot_bytes + row_off;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 v = ld_shared_v4f(src + ((uint32_t(c / 4 + q) ^ rot) << 4));
                            r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + v.x);
                            r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + v.y);
                            r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + v.z);
                            r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + v.w);
                        }
                    }
                }
                const int64_t gn0 = int64_t(nt) * tile_n + c;
                if (live && gm < M && gn0 < N) {
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
                        uint16_t* yr = static_cast<uint16_t*>(y) + gm * ldy + gn0;
                        if (vec_ok && gn0 + 32 <= N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                uint4 v;
                                v.x = pack16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), h16);
                                v.y = pack16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]), h16);
                                v.z = pack16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]), h16);
                                v.w = pack16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]), h16);
                                *reinterpret_cast<uint4*>(yr + i) = v;
                            }
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (gn0 + i < N) yr[i] = round16(__uint_as_float(r[i]), h16);
                        }
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&tempty[acc]);
            if (SPLIT) {
                // release (cluster scope) orders this thread's slot stores / slot loads
                // before the signal
                if (rank != 0) {
                    mbar_arrive_cluster(to_full);
                } else {
                    for (int sp = 1; sp < args.splits; ++sp)
                        mbar_arrive_cluster(cluster_map(smem_addr(red_free), uint32_t(sp)));
                }
            }
        }
    } else if (QUANT && KN) {
        // ---------------------------------------------- converters, natural layout
        // W is stored [K, N] and quantized along N (one scale per group of gs columns of a
        // row k; "Fix fp quantized matmul corruption...", the natural-layout qmm_n).  A
        // stage holds kbs K-blocks' 64*kbs rows of packed codes for the tile's columns.  The
        // two groups of four converter warps take alternate stages (as for the transposed
        // layout) and write the bf16 tile in the layout a TMA copy of bf16 W [K, N] gives
        // (N-major, atoms of KN_ATOM_N columns, KN_SWIZZLE-byte swizzle), so the MMA and
        // its K order are those of the dense KN GEMM.  A thread converts 8-column pieces
        // (k-row kr, columns 8c8 ..): the same per-element arithmetic as the transposed
        // layout.  Rows past K and columns past N become zeros; scales are read only for
        // elements inside W, one iteration ahead.
        constexpr int PPR = NSUB * BN / 8;       // 8-column pieces per k-row
        constexpr int NP = BK * PPR / 128;       // pieces per thread per K-block
        constexpr int MAXK = qkn_max_kbs(NSUB);  // K-blocks per stage, at most
        static_assert(NP >= 1 && (BK * PPR) % 128 == 0, "pieces per converter thread");
        const int cgrp = (warp - 6) >> 2;
        const int ct = ((warp - 6) & 3) * 32 + lane;  // 0..127 within the group
        const uint8_t* qs8 = static_cast<const uint8_t*>(args.qscales);
        const uint16_t* qs16 = static_cast<const uint16_t*>(args.qscales);
        const int nkb_t = kb1 - kb0;
        const int spt = (nkb_t + kbs - 1) / kbs;  // stages per tile
        const int tiles_mine = first_tile < num_tiles
                                   ? (num_tiles - 1 - first_tile) / tile_step + 1 : 0;
        const int iters = tiles_mine * spt;
        if (!args.w_early) pdl_wait();  // scales may come from the previous grid
        bool ok = true;
        auto run = [&](auto tag) {
            constexpr int F = decltype(tag)::value;
            constexpr bool AFF = F >= 3;
            constexpr bool EIGHT = F == 2 || F == 4;
            constexpr int RB = EIGHT ? NSUB * BN : NSUB * BN / 2;  // code bytes per k-row
            // raw scale (and bias) codes of stage j's pieces, K-block by K-block
            auto fetch = [&](int j, uint32_t (&sc)[MAXK][NP], uint32_t (&bs)[MAXK][NP]) {
                const int t = first_tile + (j / spt) * tile_step;
                const int kbf = kb0 + (j % spt) * kbs;
                const int n0 = (t % n_tiles) * tile_n;
#pragma unroll
                for (int kk = 0; kk < MAXK; ++kk) {
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        const int pc = ct + 128 * i;
                        const int k = (kbf + kk) * BK + pc / PPR;
                        const int n = n0 + (pc % PPR) * 8;
                        sc[kk][i] = 0u;
                        bs[kk][i] = 0u;
                        if (kk < kbs && kbf + kk < kb1 && k < K && n < N) {
                            const int64_t gi = int64_t(n >> gsh);
                            if (AFF) {
                                sc[kk][i] = __ldg(qs16 + int64_t(k) * args.lds + gi);
                                bs[kk][i] = __ldg(args.qbiases + int64_t(k) * args.ldb + gi);
                            } else {
                                sc[kk][i] = __ldg(qs8 + int64_t(k) * args.lds + gi);
                            }
                        }
                    }
                }
            };
            uint32_t sc[MAXK][NP] = {}, bs[MAXK][NP] = {};
            if (cgrp < iters) fetch(cgrp, sc, bs);
            uint32_t stage = uint32_t(cgrp), phase = 0;
            uint32_t wb = uint32_t(cgrp), wphase = 0;
            for (int j = cgrp; j < iters; j += 2) {
                uint32_t nsc[MAXK][NP] = {}, nbs[MAXK][NP] = {};
                if (j + 2 < iters) fetch(j + 2, nsc, nbs);
                const int t = first_tile + (j / spt) * tile_step;
                const int kbf = kb0 + (j % spt) * kbs;      // the stage's first K-block
                const int nk = kb1 - kbf < kbs ? kb1 - kbf : kbs;
                const int n0 = (t % n_tiles) * tile_n;
                if (!mbar_wait_warp(&full[stage], phase, abort_flag, wait_ns) ||
                    !mbar_wait_warp(&wfree[wb], wphase ^ 1u, abort_flag, wait_ns)) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = sR + stage * r_bytes;
                uint8_t* wt = sB + wb * kbs * b_bytes;
#pragma unroll
                for (int kk = 0; kk < MAXK; ++kk) {
                    if (kk >= nk) break;
                    const int kb = kbf + kk;
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        const int pc = ct + 128 * i;
                        const int kr = pc / PPR, c8 = pc % PPR;
                        const bool live = kb * BK + kr < K && n0 + 8 * c8 < N;
                        const uint8_t* crow = raw + (kk * BK + kr) * RB;
                        uint32_t cw[2];
                        if (EIGHT) {
                            const uint2 u = *reinterpret_cast<const uint2*>(crow + 8 * c8);
                            cw[0] = u.x;
                            cw[1] = u.y;
                        } else {
                            cw[0] = *reinterpret_cast<const uint32_t*>(crow + 4 * c8);
                            cw[1] = 0u;
                        }
                        float scf;
                        if (F == 0 || F == 2) scf = dec_e8m0(sc[kk][i]);
                        else if (F == 1) scf = dec_e4m3(sc[kk][i]);
                        else scf = widen16(uint16_t(sc[kk][i]), false);
                        const float bsf = AFF ? widen16(uint16_t(bs[kk][i]), false) : 0.f;
                        uint4 pk;
                        if (F == 0 || F == 1) {
                            uint32_t o[4];
                            e2m1x8_to_bf16(cw[0], o);
                            const uint32_t s2 = (__float_as_uint(scf) >> 16) * 0x10001u;
                            pk.x = live ? mul_bf16x2(o[0], s2) : 0u;
                            pk.y = live ? mul_bf16x2(o[1], s2) : 0u;
                            pk.z = live ? mul_bf16x2(o[2], s2) : 0u;
                            pk.w = live ? mul_bf16x2(o[3], s2) : 0u;
                        } else {
                            float v[8];
                            if (live) {
                                if (F == 2) {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const uint32_t pair = (cw[e >> 1] >> (16 * (e & 1))) & 0xffffu;
                                        const float2 f = h2_to_f2(cvt_e4m3x2(pair));
                                        v[2 * e] = f.x * scf;
                                        v[2 * e + 1] = f.y * scf;
                                    }
                                } else if (F == 4) {
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        v[e] = fmaf(scf, byte_to_f32(cw[e >> 2], e & 3), bsf);
                                } else {
                                    const uint32_t ev = cw[0] & 0x0f0f0f0fu;
                                    const uint32_t od = (cw[0] >> 4) & 0x0f0f0f0fu;
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        v[e] = fmaf(scf, byte_to_f32(e & 1 ? od : ev, e >> 1), bsf);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) v[e] = 0.f;
                            }
                            pk.x = pack_bf16x2(v[0], v[1]);
                            pk.y = pack_bf16x2(v[2], v[3]);
                            pk.z = pack_bf16x2(v[4], v[5]);
                            pk.w = pack_bf16x2(v[6], v[7]);
                        }
                        // atom c8 / (KN_ATOM_N / 8) (atoms kbs K-blocks apart), K-block kk,
                        // k-row kr (KN_SWIZZLE bytes), 16-byte piece c8 % (KN_ATOM_N / 8)
                        // under the swizzle a TMA copy applies
                        constexpr int PA = KN_ATOM_N / 8;  // pieces per atom row
                        const int pa = c8 % PA;
                        const int sw = KN_SWIZZLE == 128 ? (kr & 7) : ((kr >> 1) & 3);
                        *reinterpret_cast<uint4*>(wt + ((c8 / PA) * kbs + kk) * KN_ATOM_BYTES +
                                                  kr * KN_SWIZZLE + ((pa ^ sw) << 4)) = pk;
                    }
                }
                fence_proxy_async_smem();  // generic writes, read by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv[wb]);
                stage += 2;
                if (stage >= uint32_t(S)) {
                    stage -= uint32_t(S);
                    phase ^= 1u;
                }
                wb += 2;
                if (wb >= uint32_t(args.wbufs)) {
                    wb -= uint32_t(args.wbufs);
                    wphase ^= 1u;
                }
#pragma unroll
                for (int kk = 0; kk < MAXK; ++kk)
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        sc[kk][i] = nsc[kk][i];
                        bs[kk][i] = nbs[kk][i];
                    }
            }
        };
        switch (args.qfmt) {
            case 0: run(std::integral_constant<int, 0>{}); break;
            case 1: run(std::integral_constant<int, 1>{}); break;
            case 2: run(std::integral_constant<int, 2>{}); break;
            case 3: run(std::integral_constant<int, 3>{}); break;
            default: run(std::integral_constant<int, 4>{}); break;
        }
        if (!ok && lane == 0 && !*abort_flag) fail();
    } else if (QUANT) {
        // --------------------------------------------------------------- converters
        // Two groups of four converter warps turn the stages' packed codes into the bf16 W
        // tiles the MMA reads (K-major, 128-byte swizzle: the layout a TMA copy of bf16 W
        // would give), once a stage's copies have landed and the tile buffer is free.
        // Group g takes the iterations i = g mod 2; the ring and the buffer ring both have
        // an even length, so a group takes every use of its stages and buffers in order and
        // waits on each barrier one phase at a time.  A group's 128 threads split each
        // K-block row into PARTS parts: tiles of 64 rows or more in two halves of 64
        // threads (a warp pair each; thread ct of half h converts columns 32h..32h+31 of
        // tile rows ct, ct+64, ...), 32-row tiles in four quarters of 32 (a warp each;
        // lane ct converts columns 16h..16h+15 of row ct).  Without staged scales, a thread's
        // scales (and biases) for its next stage are loaded from global memory before it
        // waits for the current one.  Every dequantized value except the affine ones is
        // exact in bf16; affine is fmaf(scale, q, bias) rounded to bf16.  Rows past N and
        // columns past K become zeros.
        constexpr int PARTS = NSUB * BN >= 64 ? 2 : 4;        // threads per tile row
        constexpr int QR = NSUB * BN >= 64 ? NSUB * BN / 64 : 1;  // rows per thread
        // a group of GW warps: GW / 4 sets of four, set `sub` taking the stage's K-blocks
        // ki with ki mod SUBS == sub (each set covers every row and part of a K-block)
        constexpr int GW = conv_warps(KN, NSUB) / 2, SUBS = GW / 4;
        const int cgrp = (warp - 6) / GW;
        const int sub = ((warp - 6) % GW) >> 2;
        const int w4 = (warp - 6) & 3;
        // the part: for quarters, lane ct of the group's warp w takes quarter (w + ct) mod 4,
        // so a warp's lanes read four different 8-byte columns of their rows (the rows of a
        // code stage are a multiple of 128 bytes apart: one column would put every lane on
        // the same banks) and the four warps still cover every (row, quarter) once
        const int half = PARTS == 2 ? (w4 >> 1) & 1 : (w4 + lane) & 3;
        const int ct = PARTS == 2 ? (w4 & 1) * 32 + lane : lane;
        const uint8_t* qs8 = static_cast<const uint8_t*>(args.qscales);
        const uint16_t* qs16 = static_cast<const uint16_t*>(args.qscales);
        const int nkb_t = kb1 - kb0;
        const int spt = (nkb_t + kbs - 1) / kbs;  // stages per tile
        const int tiles_mine = first_tile < num_tiles
                                   ? (num_tiles - 1 - first_tile) / tile_step + 1 : 0;
        const int iters = tiles_mine * spt;
        const bool staged = args.q_staged != 0;
        if (!args.w_early) pdl_wait();  // scales may come from the previous grid
        bool ok = true;
        // one specialised loop per format (the format is uniform over the launch)
        auto run = [&](auto tag) {
            constexpr int F = decltype(tag)::value;
            constexpr bool AFF = F >= 3;
            constexpr int G = F == 1 ? 4 : 2;  // scale segments per K-block row
            constexpr int SEG = BK / G;        // columns per segment (<= the group size)
            constexpr int PP = 8 / PARTS;      // 8-column pieces per part
            constexpr int GH = (PP * 8 + SEG - 1) / SEG;  // segments a part spans
            constexpr int RW = (F == 2 || F == 4) ? BK / 4 : BK / 8;  // code words per row
            constexpr int HW = RW / PARTS;     // ... per part
            const int seg0 = (half * PP * 8) / SEG;  // the part's first segment
            // raw scale (and bias) codes of iteration j's rows, one per segment of the half
            auto fetch = [&](int j, uint32_t (&sc)[QR][GH], uint32_t (&bs)[QR][GH]) {
                const int t = first_tile + (j / nkb_t) * tile_step;  // (kbs = 1 here)
                const int kb = kb0 + j % nkb_t;
                const int n0 = (t % n_tiles) * tile_n;
#pragma unroll
                for (int q = 0; q < QR; ++q) {
                    const int n = n0 + ct + 64 * q;
#pragma unroll
                    for (int gg = 0; gg < GH; ++gg) {
                        const int k = kb * BK + (seg0 + gg) * SEG;
                        sc[q][gg] = 0u;
                        bs[q][gg] = 0u;
                        if (n < N && k < K) {
                            const int64_t gi = int64_t(k >> gsh);
                            if (AFF) {
                                sc[q][gg] = __ldg(qs16 + int64_t(n) * args.lds + gi);
                                bs[q][gg] = __ldg(args.qbiases + int64_t(n) * args.ldb + gi);
                            } else {
                                sc[q][gg] = __ldg(qs8 + int64_t(n) * args.lds + gi);
                            }
                        }
                    }
                }
            };
            uint32_t sc[QR][GH] = {}, bs[QR][GH] = {};
            if (!staged && cgrp < iters) fetch(cgrp, sc, bs);
            uint32_t stage = uint32_t(cgrp), phase = 0;
            uint32_t wb = uint32_t(cgrp), wphase = 0;
            for (int j = cgrp; j < iters; j += 2) {
                uint32_t nsc[QR][GH] = {}, nbs[QR][GH] = {};
                if (!staged && j + 2 < iters) fetch(j + 2, nsc, nbs);
                const int t = first_tile + (j / spt) * tile_step;
                const int kbf = kb0 + (j % spt) * kbs;      // the stage's first K-block
                const int nk = kb1 - kbf < kbs ? kb1 - kbf : kbs;
                const int n0 = (t % n_tiles) * tile_n;
                if (!mbar_wait_warp(&full[stage], phase, abort_flag, wait_ns) ||
                    !mbar_wait_warp(&wfree[wb], wphase ^ 1u, abort_flag, wait_ns)) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = sR + stage * r_bytes;
                // the staged scale window starts at the 16-byte boundary at or below the
                // stage's first group
                const int xs = ((kbf * BK) >> gsh) & ~(s_epb - 1);
#pragma unroll 1
                for (int ki = sub; ki < nk; ki += SUBS) {  // the stage's K-blocks (this set's)
                const int kb = kbf + ki;
                uint8_t* wt = sB + (wb * kbs + ki) * b_bytes;
                if (staged) {  // this K-block's scales (and biases) from shared memory
                    const uint8_t* ss = raw + codes_bytes;
#pragma unroll
                    for (int q = 0; q < QR; ++q) {
                        const int r = ct + 64 * q;
#pragma unroll
                        for (int gg = 0; gg < GH; ++gg) {
                            const int gi = ((kb * BK + (seg0 + gg) * SEG) >> gsh) - xs;
                            if (AFF) {
                                sc[q][gg] = reinterpret_cast<const uint16_t*>(ss)[r * (s_row / 2) + gi];
                                bs[q][gg] = reinterpret_cast<const uint16_t*>(ss + s_blk)[r * (s_row / 2) + gi];
                            } else {
                                sc[q][gg] = ss[r * s_row + gi];
                            }
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < QR; ++q) {
                    const int r = ct + 64 * q;
                    const bool row_live = n0 + r < N;
                    uint32_t cw[HW];  // the code words of this part of the row
                    const uint8_t* crow = raw + r * (kbs * RW * 4) + ki * (RW * 4) + half * (HW * 4);
                    if constexpr (HW >= 4) {
#pragma unroll
                        for (int i = 0; i < HW / 4; ++i) {
                            const uint4 u = *reinterpret_cast<const uint4*>(crow + 16 * i);
                            cw[4 * i] = u.x;
                            cw[4 * i + 1] = u.y;
                            cw[4 * i + 2] = u.z;
                            cw[4 * i + 3] = u.w;
                        }
                    } else {
                        const uint2 u = *reinterpret_cast<const uint2*>(crow);
                        cw[0] = u.x;
                        cw[1 % HW] = u.y;
                    }
                    float scf[GH], bsf[GH];
#pragma unroll
                    for (int gg = 0; gg < GH; ++gg) {
                        if (F == 0 || F == 2) scf[gg] = dec_e8m0(sc[q][gg]);
                        else if (F == 1) scf[gg] = dec_e4m3(sc[q][gg]);
                        else scf[gg] = widen16(uint16_t(sc[q][gg]), false);
                        bsf[gg] = AFF ? widen16(uint16_t(bs[q][gg]), false) : 0.f;
                    }
                    uint8_t* wrow = wt + q * (64 * BK * 2) + (ct >> 3) * 1024 + (ct & 7) * 128;
#pragma unroll
                    for (int pp = 0; pp < PP; ++pp) {  // 8-column pieces (16 bytes of bf16)
                        const int p = PP * half + pp;
                        // the piece's segment within the part (the part starts on a
                        // segment boundary, or -- quarters of 32-column segments -- inside
                        // one): known at compile time
                        const int gg = PARTS == 2 ? (8 * pp) / SEG : 0;
                        const bool live = row_live && kb * BK + 8 * p < K;  // K % 16 == 0
                        uint4 pk;
                        if (F == 0 || F == 1) {
                            // FP4 E2M1 codes times the block scale, in bf16: every product
                            // is exact in bf16 (or overflows), so bf16 arithmetic rounds
                            // nothing
                            uint32_t o[4];
                            e2m1x8_to_bf16(cw[pp], o);
                            const uint32_t s2 = (__float_as_uint(scf[gg]) >> 16) * 0x10001u;
                            pk.x = live ? mul_bf16x2(o[0], s2) : 0u;
                            pk.y = live ? mul_bf16x2(o[1], s2) : 0u;
                            pk.z = live ? mul_bf16x2(o[2], s2) : 0u;
                            pk.w = live ? mul_bf16x2(o[3], s2) : 0u;
                            *reinterpret_cast<uint4*>(wrow + ((p ^ (ct & 7)) << 4)) = pk;
                            continue;
                        }
                        const float s = scf[gg], b = bsf[gg];
                        float v[8];
                        if (live) {
                            if (F == 2) {  // FP8 E4M3 codes times the block scale
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const uint32_t pair = (cw[2 * pp + (e >> 1)] >> (16 * (e & 1))) & 0xffffu;
                                    const float2 f = h2_to_f2(cvt_e4m3x2(pair));
                                    v[2 * e] = f.x * s;
                                    v[2 * e + 1] = f.y * s;
                                }
                            } else if (F == 4) {  // affine 8-bit: fmaf(scale, q, bias)
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    v[e] = fmaf(s, byte_to_f32(cw[2 * pp + (e >> 2)], e & 3), b);
                            } else {  // affine 4-bit: nibbles spread to bytes first
                                const uint32_t ev = cw[pp] & 0x0f0f0f0fu, od = (cw[pp] >> 4) & 0x0f0f0f0fu;
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    v[e] = fmaf(s, byte_to_f32(e & 1 ? od : ev, e >> 1), b);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = 0.f;
                        }
                        pk.x = pack_bf16x2(v[0], v[1]);
                        pk.y = pack_bf16x2(v[2], v[3]);
                        pk.z = pack_bf16x2(v[4], v[5]);
                        pk.w = pack_bf16x2(v[6], v[7]);
                        *reinterpret_cast<uint4*>(wrow + ((p ^ (ct & 7)) << 4)) = pk;
                    }
                }
                }  // K-blocks of the stage
                fence_proxy_async_smem();  // generic writes, read by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv[wb]);
                stage += 2;  // S and wbufs are even: the group stays on its own stages
                if (stage >= uint32_t(S)) {  // and buffers
                    stage -= uint32_t(S);
                    phase ^= 1u;
                }
                wb += 2;
                if (wb >= uint32_t(args.wbufs)) {
                    wb -= uint32_t(args.wbufs);
                    wphase ^= 1u;
                }
#pragma unroll
                for (int q = 0; q < QR; ++q)
#pragma unroll
                    for (int gg = 0; gg < GH; ++gg) {
                        sc[q][gg] = nsc[q][gg];
                        bs[q][gg] = nbs[q][gg];
                    }
            }
        };
        switch (args.qfmt) {
            case 0: run(std::integral_constant<int, 0>{}); break;
            case 1: run(std::integral_constant<int, 1>{}); break;
            case 2: run(std::integral_constant<int, 2>{}); break;
            case 3: run(std::integral_constant<int, 3>{}); break;
            default: run(std::integral_constant<int, 4>{}); break;
        }
        if (!ok && lane == 0 && !*abort_flag) fail();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    // no CTA leaves while another CTA of its cluster may still signal its barriers or
    // write its shared memory (every loop above ends, by completion or by timeout)
    if constexpr (SPLIT) cluster_sync_all();
}

template <bool KN, bool F32OUT, int NSUB, int MSUB = 1>
cudaError_t launch_t(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                     const GemmArgs& a, int grid, cudaStream_t s) {
    auto kern = gemm_kernel<KN, F32OUT, NSUB, false, MSUB, false>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(THREADS), SMEM_BYTES, s, mx, mw, mw, mw, a,
                      dev.err_word);
}

// The split-K kernel: clusters of a.splits CTAs, as many clusters as fit on the GPU at
// once (cluster placement is limited by the GPCs, so this can be fewer than SMs/splits),
// never more than there are tiles.
template <bool KN, bool F32OUT>
cudaError_t launch_split(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                         const GemmArgs& a, int64_t tiles, cudaStream_t s) {
    auto kern = gemm_kernel<KN, F32OUT, 1, true, 1, false>;
    static bool attr_done[64] = {};
    static int fit[64][MAX_SPLITS + 1] = {};  // co-resident clusters per device and size
    if (dev.device < 0 || dev.device >= 64 || a.splits < 2 || a.splits > MAX_SPLITS)
        return cudaErrorNotSupported;
    if (!attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    int& n_fit = fit[dev.device][a.splits];
    if (n_fit == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(a.splits));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(a.splits);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorNotSupported;
        n_fit = n;
    }
    const int clusters = int(tiles < n_fit ? tiles : n_fit);
    return launch_pdl_cluster(kern, dim3(unsigned(clusters * a.splits)), dim3(THREADS),
                              SMEM_BYTES, s, unsigned(a.splits), mx, mw, mw, mw, a, dev.err_word);
}

template <bool F32OUT, int NSUB, bool KN = false>
cudaError_t launch_q(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                     const CUtensorMap& ms, const CUtensorMap& mb, const GemmArgs& a, int grid,
                     cudaStream_t s) {
    auto kern = gemm_kernel<KN, F32OUT, NSUB, false, 1, true>;
    static bool attr_done[64] = {};
    if (dev.device >= 0 && dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev.device] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(gemm_threads(true, KN, NSUB)), SMEM_BYTES, s, mx,
                      mw, ms, mb, a, dev.err_word);
}

template <bool KN, bool F32OUT>
cudaError_t launch_nsub(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                        const GemmArgs& a, int grid, cudaStream_t s) {
    switch (a.nsub) {
        case 1: return launch_t<KN, F32OUT, 1>(dev, mx, mw, a, grid, s);
        case 2: return launch_t<KN, F32OUT, 2>(dev, mx, mw, a, grid, s);
        case 4: return launch_t<KN, F32OUT, 4>(dev, mx, mw, a, grid, s);
        default:
            if (a.a_rows == 2 * BM)  // two instruction tiles along M per CTA tile
                return launch_t<KN, F32OUT, MAX_NSUB, 2>(dev, mx, mw, a, grid, s);
            return launch_t<KN, F32OUT, MAX_NSUB>(dev, mx, mw, a, grid, s);
    }
}

}  // namespace

int gemm_tile_n() { return BN; }

GemmSchedule gemm_schedule(int64_t M, int64_t N, int64_t K, bool w_kn, int num_sms,
                           bool split_ok) {
    GemmSchedule g;
    const int64_t m_tiles = (M + BM - 1) / BM;
    const int64_t nkb = (K + BK - 1) / BK;
    g.a_rows = m_tiles == 1 ? int((M + 7) / 8 * 8) : BM;
    // CTA tile shape from a cost model: per K-block a CTA spends the longer of its MMAs
    // (about 8192 flop per cycle per SM) and its operand copies (about 64 bytes per cycle
    // per SM from L2), and the tiles run in ceil(tiles / SMs) waves.  Candidates: 128 x
    // BN*nsub (32 to 256 columns) and 256 x 256 (two instruction tiles along M); the
    // widest wins ties (X and W are re-read from L2 the fewest times).  The instructions
    // and their K order are the same for every shape.
    const int single_rows = g.a_rows;
    double best = 0.0;
    bool wide_m = false;
    for (int msub = 2; msub >= 1; --msub) {
        for (int ns = MAX_NSUB; ns >= 1; ns >>= 1) {
            if (msub == 2 && (ns != MAX_NSUB || m_tiles < 2)) continue;
            const int64_t tm = int64_t(BM) * msub;
            const int64_t tiles = ((M + tm - 1) / tm) * ((N + int64_t(ns) * BN - 1) / (int64_t(ns) * BN));
            const int64_t waves = (tiles + num_sms - 1) / num_sms;
            const int64_t rows = msub == 2 ? tm : (m_tiles == 1 ? single_rows : BM);
            const double mma = double(msub) * ns * BM * BN * BK * 2 / 8192.0;
            const double copy = (double(rows) * BK * 2 + double(ns) * B_KB_BYTES) / 64.0;
            const double cost = double(waves) * double(nkb) * (mma > copy ? mma : copy);
            if (best == 0.0 || cost < best) {
                best = cost;
                g.nsub = ns;
                wide_m = msub == 2;
            }
        }
    }
    if (wide_m) g.a_rows = 2 * BM;
    g.kn_wide = w_kn && (g.nsub * BN >= DKN_ATOM_N || g.a_rows <= DKN_MAX_ROWS) ? 1 : 0;
    const int w_kb = g.kn_wide ? dkn_cols(g.nsub) * BK * 2 : g.nsub * B_KB_BYTES;
    // Split-K (non-invariant kernel only): a single M-tile whose instruction tiles leave
    // SMs idle gets a cluster of CTAs per tile, each over a contiguous K range, so more
    // SMs stream W and each runs a shorter chain of dependent MMAs.  The reduction slots
    // come out of the ring.
    g.splits = 1;
    g.ring_bytes = RING_BYTES;
    if (split_ok && m_tiles == 1 && g.nsub == 1) {
        int64_t sp = num_sms / ((N + BN - 1) / BN);
        if (sp > MAX_SPLITS) sp = MAX_SPLITS;
        if (sp > nkb) sp = nkb;
        // the ring keeps room for at least four stages of one K-block
        const int64_t slot = int64_t(g.a_rows) * BN * 4;
        const int64_t blk1 = int64_t(g.a_rows) * BK * 2 + w_kb;
        while (sp >= 2 && RING_BYTES - (sp - 1) * slot < 4 * blk1) --sp;
        if (sp >= 2) {
            g.splits = int(sp);
            g.ring_bytes = RING_BYTES - (g.splits - 1) * g.a_rows * BN * 4;
        }
    }
    // as many K-blocks per stage as keep at least four stages in the ring (fewer
    // barrier round trips per MMA) -- and, when split, at least four stages per CTA
    const int blk_bytes = g.a_rows * BK * 2 + w_kb;
    const int64_t per_cta = (nkb + g.splits - 1) / g.splits;
    g.kbs = 1;
    for (int kbs = w_kn ? MAX_KBS_KN : MAX_KBS; kbs >= 2; kbs >>= 1) {
        if (g.ring_bytes / (kbs * blk_bytes) >= 4 && (g.splits == 1 || per_cta >= 4 * kbs)) {
            g.kbs = kbs;
            break;
        }
    }
    g.stages = g.ring_bytes / (g.kbs * blk_bytes);
    if (g.stages > MAX_STAGES) g.stages = MAX_STAGES;
    g.kb_per_split = int(nkb);
    if (g.splits > 1) {
        const int64_t per = (per_cta + g.kbs - 1) / g.kbs * g.kbs;  // whole stages per CTA
        g.splits = int((nkb + per - 1) / per);                     // no CTA without work
        g.kb_per_split = int(per);
    }
    g.tiles = (wide_m ? (M + 2 * BM - 1) / (2 * BM) : m_tiles) *
              ((N + int64_t(g.nsub) * BN - 1) / (int64_t(g.nsub) * BN));
    g.blocked = (K % BK) == 0 ? 1 : 0;
    return g;
}

cudaError_t launch_gemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* w,
                        int64_t ldw, bool w_kn, void* y, int64_t ldy, bool y_f32, int64_t M,
                        int64_t N, int64_t K, bool split_ok, bool f16, bool w_early,
                        cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0) {
        // an empty reduction: every output is +0 (all-zero bits in bf16, binary16 and fp32)
        const size_t es = y_f32 ? 4 : 2;
        return cudaMemset2DAsync(y, size_t(ldy) * es, 0, size_t(N) * es, size_t(M), stream);
    }
    const GemmSchedule g = gemm_schedule(M, N, K, w_kn, dev.num_sms, split_ok);
    // an MMA reads A_MMA_BYTES from the start of its X block: the last X block's read must
    // stay inside the ring (it runs into the W blocks that follow the X blocks)
    const int64_t a_bytes = int64_t(g.a_rows) * BK * 2;
    const int64_t blocks = int64_t(g.stages) * g.kbs;
    const int64_t a_read = g.a_rows > BM ? a_bytes : A_MMA_BYTES;  // from an X block's start
    const int64_t w_blk = g.kn_wide ? int64_t(dkn_cols(g.nsub)) * BK * 2 : int64_t(g.nsub) * B_KB_BYTES;
    if ((blocks - 1) * a_bytes + a_read > blocks * (a_bytes + w_blk) ||
        blocks * (a_bytes + w_blk) > g.ring_bytes || g.stages < 2)
        return cudaErrorNotSupported;
    CUtensorMap mx, mw;
    bool ok;
    if (g.blocked)
        ok = tmap_kblocked_bf16(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK,
                                uint32_t(g.a_rows), uint32_t(g.kbs), 128, f16);
    else
        ok = tmap_2d_bf16(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK, uint32_t(g.a_rows),
                          128, f16);
    if (!ok) return cudaErrorNotSupported;
    if (w_kn)
        ok = tmap_2d_bf16(&mw, w, uint64_t(N), uint64_t(K), uint64_t(ldw),
                          g.kn_wide ? DKN_ATOM_N : KN_ATOM_N, uint32_t(BK * g.kbs),
                          g.kn_wide ? DKN_ATOM_N * 2 : KN_SWIZZLE, f16);
    else if (g.blocked)
        ok = tmap_kblocked_bf16(&mw, w, uint64_t(K), uint64_t(N), uint64_t(ldw), BK,
                                uint32_t(g.nsub * BN), uint32_t(g.kbs), 128, f16);
    else
        ok = tmap_2d_bf16(&mw, w, uint64_t(K), uint64_t(N), uint64_t(ldw), BK,
                          uint32_t(g.nsub * BN), 128, f16);
    if (!ok) return cudaErrorNotSupported;
    GemmArgs a{};
    a.y = y;
    a.ldy = ldy;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.a_rows = g.a_rows;
    a.nsub = g.nsub;
    a.kbs = g.kbs;
    a.blocked = g.blocked;
    a.stages = g.stages;
    a.w_stream_once = (M + BM - 1) / BM == 1 ? 1 : 0;
    a.w_early = w_early ? 1 : 0;
    a.splits = g.splits;
    a.kb_per_split = g.kb_per_split;
    a.f16 = f16 ? 1 : 0;
    a.kn_wide = g.kn_wide;
    if (g.splits > 1)
        return w_kn ? (y_f32 ? launch_split<true, true>(dev, mx, mw, a, g.tiles, stream)
                             : launch_split<true, false>(dev, mx, mw, a, g.tiles, stream))
                    : (y_f32 ? launch_split<false, true>(dev, mx, mw, a, g.tiles, stream)
                             : launch_split<false, false>(dev, mx, mw, a, g.tiles, stream));
    const int grid = int(g.tiles < dev.num_sms ? g.tiles : dev.num_sms);
    if (w_kn)
        return y_f32 ? launch_nsub<true, true>(dev, mx, mw, a, grid, stream)
                     : launch_nsub<true, false>(dev, mx, mw, a, grid, stream);
    return y_f32 ? launch_nsub<false, true>(dev, mx, mw, a, grid, stream)
                 : launch_nsub<false, false>(dev, mx, mw, a, grid, stream);
}

// Quantized W in the natural layout: codes [K, N] (row k: N codes, packed bytes, row
// stride ldq), quantized along N (scales [K, N/gs], row stride lds; biases likewise).
// The scales are read by the converters, one stage ahead.  One M-tile (small M): stages
// of several K-blocks (one code box of 64*kbs rows), so the per-stage copies, barriers
// and commits are paid once per several K-blocks.
cudaError_t launch_qgemm_kn(const DeviceInfo& dev, const void* x, int64_t ldx, const void* wq,
                            int64_t ldq, const void* scales, int64_t lds, const void* biases,
                            int64_t ldb, int fmt, int gs, void* y, int64_t ldy, bool y_f32,
                            int64_t M, int64_t N, int64_t K, bool w_early, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0) {
        const size_t es = y_f32 ? 4 : 2;
        return cudaMemset2DAsync(y, size_t(ldy) * es, 0, size_t(N) * es, size_t(M), stream);
    }
    const int64_t m_tiles = (M + BM - 1) / BM;
    const int a_rows = m_tiles == 1 ? int((M + 7) / 8 * 8) : BM;
    int nsub = 1;  // the widest tile that still gives every SM a tile
    for (int ns = MAX_NSUB; ns > 1; ns >>= 1) {
        if (m_tiles * ((N + int64_t(ns) * BN - 1) / (int64_t(ns) * BN)) >= dev.num_sms) {
            nsub = ns;
            break;
        }
    }
    const bool eight = fmt == 2 || fmt == 4;
    const int q_kb_bytes = eight ? BK : BK / 2;  // code bytes per 64 elements
    const int64_t a_bytes = int64_t(a_rows) * BK * 2;
    auto plan = [&](int k, int& wbufs_out, int& stages_out) {
        const int64_t blk = k * (a_bytes + int64_t(nsub) * BN * q_kb_bytes);  // X + codes
        const int64_t bb = int64_t(k) * nsub * B_KB_BYTES;                    // bf16 W tiles
        wbufs_out = stages_out = 0;
        for (int wb = MAX_QWBUF; wb >= 2; wb -= 2) {
            int st = int((RING_BYTES - wb * bb) / blk);
            if (st > MAX_QSTAGES) st = MAX_QSTAGES;
            st &= ~1;  // even: each converter group owns every other stage
            if (st >= 4 || (wb == 2 && st >= 2)) {
                wbufs_out = wb;
                stages_out = st;
                return;
            }
        }
    };
    int kbs = 1, wbufs = 0, stages = 0;
    if (m_tiles == 1) {
        const int64_t nkb = (K + BK - 1) / BK;
        for (kbs = qkn_max_kbs(int(nsub)); kbs > 1 && nkb < 4 * kbs; kbs >>= 1) {
        }  // keep >= 4 stages per tile
        for (; kbs > 1; kbs >>= 1) {  // and a ring of >= 4 stages
            plan(kbs, wbufs, stages);
            if (stages >= 4) break;
        }
    }
    plan(kbs, wbufs, stages);
    const int64_t bb = int64_t(kbs) * nsub * B_KB_BYTES;
    if (wbufs == 0 || (int64_t(stages) * kbs - 1) * a_bytes + A_MMA_BYTES >
                          int64_t(stages) * kbs * a_bytes + wbufs * bb)
        return cudaErrorNotSupported;
    CUtensorMap mx, mw;
    if (!tmap_2d_bf16(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK, uint32_t(a_rows), 128) ||
        !tmap_2d_u8(&mw, wq, uint64_t(eight ? N : N / 2), uint64_t(K), uint64_t(ldq),
                    uint32_t(eight ? nsub * BN : nsub * BN / 2), uint32_t(kbs * BK)))
        return cudaErrorNotSupported;
    GemmArgs a{};
    a.y = y;
    a.ldy = ldy;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.a_rows = a_rows;
    a.nsub = nsub;
    a.kbs = kbs;
    a.blocked = 0;
    a.stages = stages;
    a.w_stream_once = m_tiles == 1 ? 1 : 0;
    a.w_early = w_early ? 1 : 0;
    a.splits = 1;
    a.kb_per_split = int((K + BK - 1) / BK);
    a.f16 = 0;
    a.qfmt = fmt;
    a.gs = gs;
    a.qscales = scales;
    a.lds = lds;
    a.qbiases = static_cast<const uint16_t*>(biases);
    a.ldb = ldb;
    a.q_kb_bytes = q_kb_bytes;
    a.wbufs = wbufs;
    a.q_staged = 0;
    a.q_srow = Q_SROW;
    const int64_t tiles = m_tiles * ((N + int64_t(nsub) * BN - 1) / (int64_t(nsub) * BN));
    const int grid = int(tiles < dev.num_sms ? tiles : dev.num_sms);
    switch (nsub) {
        case 1: return y_f32 ? launch_q<true, 1, true>(dev, mx, mw, mw, mw, a, grid, stream)
                             : launch_q<false, 1, true>(dev, mx, mw, mw, mw, a, grid, stream);
        case 2: return y_f32 ? launch_q<true, 2, true>(dev, mx, mw, mw, mw, a, grid, stream)
                             : launch_q<false, 2, true>(dev, mx, mw, mw, mw, a, grid, stream);
        case 4: return y_f32 ? launch_q<true, 4, true>(dev, mx, mw, mw, mw, a, grid, stream)
                             : launch_q<false, 4, true>(dev, mx, mw, mw, mw, a, grid, stream);
        default: return y_f32 ? launch_q<true, MAX_NSUB, true>(dev, mx, mw, mw, mw, a, grid, stream)
                              : launch_q<false, MAX_NSUB, true>(dev, mx, mw, mw, mw, a, grid, stream);
    }
}

cudaError_t launch_qgemm(const DeviceInfo& dev, const void* x, int64_t ldx, const void* wq,
                         int64_t ldq, const void* scales, int64_t lds, const void* biases,
                         int64_t ldb, int fmt, int gs, void* y, int64_t ldy, bool y_f32,
                         int64_t M, int64_t N, int64_t K, bool w_early, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    if (K == 0) {
        const size_t es = y_f32 ? 4 : 2;
        return cudaMemset2DAsync(y, size_t(ldy) * es, 0, size_t(N) * es, size_t(M), stream);
    }
    // the invariant schedule with one K-block per stage and 128-row CTA tiles
    const int64_t m_tiles = (M + BM - 1) / BM;
    const int a_rows = m_tiles == 1 ? int((M + 7) / 8 * 8) : BM;
    // tiles of 32 to 256 rows of W: the widest that still gives every SM a tile
    constexpr int QMIN = 1;
    int nsub = QMIN;
    for (int ns = MAX_NSUB; ns > QMIN; ns >>= 1) {
        if (m_tiles * ((N + int64_t(ns) * BN - 1) / (int64_t(ns) * BN)) >= dev.num_sms) {
            nsub = ns;
            break;
        }
    }
    const bool eight = fmt == 2 || fmt == 4;
    const bool aff = fmt >= 3;
    const int q_kb_bytes = eight ? BK : BK / 2;
    // Scales (and biases) travel with the codes, by TMA, when their rows start on 16-byte
    // boundaries (a tensor map's rule); else the converters load them themselves.
    const bool stageable =
        reinterpret_cast<uintptr_t>(scales) % 16 == 0 && (lds * (aff ? 2 : 1)) % 16 == 0 &&
        (!aff || (reinterpret_cast<uintptr_t>(biases) % 16 == 0 && (ldb * 2) % 16 == 0));
    // One M-tile (small M): stages of several K-blocks (a code box of at most 256 bytes a
    // row, a 64-byte scale window covering them), so the per-stage copies, barriers and
    // commits are paid once per several K-blocks; they need staged scales.
    const int64_t a_bytes = int64_t(a_rows) * BK * 2;
    // The ring's stages hold kbs X blocks and their packed codes (and the staged scales);
    // the bf16 tiles the converters write get their own buffers (kbs tiles each): four
    // when the ring can still be four stages deep, else two.
    auto plan = [&](int k, bool with_scales, int srow, int& wbufs_out, int& stages_out) {
        const int64_t blk = k * (a_bytes + int64_t(nsub) * BN * q_kb_bytes) +
                            (with_scales ? (aff ? 2 : 1) * int64_t(nsub) * BN * srow : 0);
        const int64_t bb = int64_t(k) * nsub * B_KB_BYTES;
        wbufs_out = stages_out = 0;
        for (int wb = MAX_QWBUF; wb >= 2; wb -= 2) {
            int st = int((RING_BYTES - wb * bb) / blk);
            if (st > MAX_QSTAGES) st = MAX_QSTAGES;
            st &= ~1;  // even: each of the two converter groups owns every other stage
            if (st >= 4 || (wb == 2 && st >= 2)) {
                wbufs_out = wb;
                stages_out = st;
                return;
            }
        }
    };
    int kbs = 1, wbufs = 0, stages = 0;
    if (stageable && m_tiles == 1) {
        const int64_t nkb = (K + BK - 1) / BK;
        kbs = 256 / q_kb_bytes < 8 ? 256 / q_kb_bytes : 8;
        while (kbs > 1 && nkb < 4 * kbs) kbs >>= 1;  // keep >= 4 stages per tile
        for (; kbs > 1; kbs >>= 1) {                   // and a ring of >= 4 stages
            plan(kbs, true, Q_SROW_KBS, wbufs, stages);
            if (stages >= 4) break;
        }
    }
    CUtensorMap ms, mb;
    const int64_t groups = K / gs;
    auto stage_scales = [&](int srow) {
        return aff ? tmap_2d_u16(&ms, scales, uint64_t(groups), uint64_t(N), uint64_t(lds * 2),
                                 uint32_t(srow / 2), uint32_t(nsub * BN)) &&
                         tmap_2d_u16(&mb, biases, uint64_t(groups), uint64_t(N),
                                     uint64_t(ldb * 2), uint32_t(srow / 2), uint32_t(nsub * BN))
                   : tmap_2d_u8(&ms, scales, uint64_t(groups), uint64_t(N), uint64_t(lds),
                                uint32_t(srow), uint32_t(nsub * BN));
    };
    bool staged = stageable && stage_scales(kbs > 1 ? Q_SROW_KBS : Q_SROW);
    if (!staged && kbs > 1) {  // no window of several K-blocks: one K-block per stage
        kbs = 1;
        staged = stageable && stage_scales(Q_SROW);
    }
    const int s_row = kbs > 1 ? Q_SROW_KBS : Q_SROW;
    plan(kbs, staged, s_row, wbufs, stages);
    const int64_t b_bytes = int64_t(kbs) * nsub * B_KB_BYTES;
    // an MMA reads A_MMA_BYTES from the start of its X block: the last block's read runs
    // into the tile buffers that follow the X blocks and must stay inside the ring
    if (wbufs == 0 ||
        (int64_t(stages) * kbs - 1) * a_bytes + A_MMA_BYTES > int64_t(stages) * kbs * a_bytes +
                                                                 wbufs * b_bytes)
        return cudaErrorNotSupported;
    CUtensorMap mx, mw;
    if (!tmap_2d_bf16(&mx, x, uint64_t(K), uint64_t(M), uint64_t(ldx), BK, uint32_t(a_rows), 128) ||
        !tmap_2d_u8(&mw, wq, uint64_t(eight ? K : K / 2), uint64_t(N), uint64_t(ldq),
                    uint32_t(kbs * q_kb_bytes), uint32_t(nsub * BN)))
        return cudaErrorNotSupported;
    GemmArgs a{};
    a.y = y;
    a.ldy = ldy;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.a_rows = a_rows;
    a.nsub = nsub;
    a.kbs = kbs;
    a.blocked = 0;
    a.stages = stages;
    a.w_stream_once = m_tiles == 1 ? 1 : 0;
    a.w_early = w_early ? 1 : 0;
    a.splits = 1;
    a.kb_per_split = int((K + BK - 1) / BK);
    a.f16 = 0;
    a.qfmt = fmt;
    a.gs = gs;
    a.qscales = scales;
    a.lds = lds;
    a.qbiases = static_cast<const uint16_t*>(biases);
    a.ldb = ldb;
    a.q_kb_bytes = q_kb_bytes;
    a.wbufs = wbufs;
    a.q_staged = staged ? 1 : 0;
    a.q_srow = s_row;
    if (!staged) ms = mb = mw;  // unused
    else if (!aff) mb = ms;
    const int64_t tiles = m_tiles * ((N + int64_t(nsub) * BN - 1) / (int64_t(nsub) * BN));
    const int grid = int(tiles < dev.num_sms ? tiles : dev.num_sms);
    switch (nsub) {
        case 1: return y_f32 ? launch_q<true, 1>(dev, mx, mw, ms, mb, a, grid, stream)
                             : launch_q<false, 1>(dev, mx, mw, ms, mb, a, grid, stream);
        case 2: return y_f32 ? launch_q<true, 2>(dev, mx, mw, ms, mb, a, grid, stream)
                             : launch_q<false, 2>(dev, mx, mw, ms, mb, a, grid, stream);
        case 4: return y_f32 ? launch_q<true, 4>(dev, mx, mw, ms, mb, a, grid, stream)
                             : launch_q<false, 4>(dev, mx, mw, ms, mb, a, grid, stream);
        default: return y_f32 ? launch_q<true, MAX_NSUB>(dev, mx, mw, ms, mb, a, grid, stream)
                              : launch_q<false, MAX_NSUB>(dev, mx, mw, ms, mb, a, grid, stream);
    }
}

}  // namespace bi
