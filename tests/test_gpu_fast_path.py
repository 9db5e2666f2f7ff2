"""The non-invariant fast paths, taken by calls outside the batch-invariant limit, on the
GPU: parity with the CPU oracle, run-to-run determinism, and the pages' limit experiment
("Fix/speculative shape invariance", ml-explore/mlx PR 4279, review thread: with the
limit at 0 a token computed alone and inside a block diverge, with the limit covering
the block they match; section Changes: long prefills and dimensions above the limit keep
the optimized paths)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16, check_f32, check_rows_rel_l2

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def sms(dev):
    return torch.cuda.get_device_properties(dev).multi_processor_count


# ------------------------------------------------------------------- split-K matmul

FAST_SHAPES = [
    # (M, N, K, layout); every one splits K at limit 0 on a 152-SM GPU
    (1, 2048, 4096, "nk"),      # 2 CTAs per tile
    (8, 1024, 4096, "kn"),      # 4 CTAs per tile
    (5, 1000, 4160, "nk"),      # ragged N, K tail (one copy per K-block)
    (50, 1024, 4096, "kn"),     # 56 staged rows: M = 64 instructions, four lane quarters
    (100, 1024, 4096, "nk"),    # 104 staged rows: the slots limit the split
    (128, 512, 1000, "kn"),     # a full M-tile, ragged K
    (3, 64, 4096, "nk"),        # a single column tile
]


@pytest.mark.parametrize("M,N,K,layout", FAST_SHAPES)
def test_split_k_parity(dev, sms, M, N, K, layout):
    bi.set_batch_invariant_limit(0)
    assert bi.matmul_splits(M, N, K, layout, sms) > 1
    gi = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    w = (gi.w_nk if layout == "nk" else gi.w_kn).to(dev)
    x = gi.x.to(dev)
    ref = oracle.matmul(inputs.bf16_bits(gi.x), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_bf16(bi.matmul(x, w, layout), ref, f"split-K {layout} {M}x{N}x{K}")
    y32 = bi.matmul(x, w, layout, out_dtype=torch.float32)
    X = np.abs(gi.x.float().numpy().astype(np.float64))
    W = np.abs(gi.w_nk.float().numpy().astype(np.float64))
    check_f32(y32, ref, X @ W.T, f"split-K fp32 {layout} {M}x{N}x{K}")


def test_split_k_is_deterministic_and_chains(dev):
    """Repeated calls give one result; back-to-back dependent split-K launches (each
    waiting on the previous grid) read their inputs only once those are complete."""
    bi.set_batch_invariant_limit(0)
    M, N, K = 8, 4096, 4096
    gi = inputs.gemm_inputs(M, N, K, seed=3)
    w2 = inputs.normal_bf16((1024, N), std=0.02, seed=4)      # y1 [8,4096] -> y2 [8,1024]
    w3 = inputs.normal_bf16((N, 1024), std=0.02, seed=5)      # y2 -> y3 [8,4096]
    x, w, w2d, w3d = gi.x.to(dev), gi.w_nk.to(dev), w2.to(dev), w3.to(dev)
    seen = set()
    for _ in range(20):
        seen.add(bytes(bi.matmul(x, w).view(torch.int16).cpu().numpy()))
    assert len(seen) == 1
    y1 = bi.matmul(x, w)
    for _ in range(5):  # y1 -> y2 (split) -> y3 (invariant), no synchronisation in between
        y2 = bi.matmul(y1, w2d)
        bi.set_batch_invariant_limit(1 << 20)
        y3 = bi.matmul(y2, w3d)
        bi.set_batch_invariant_limit(0)
    torch.cuda.synchronize()
    b = inputs.bf16_bits
    check_bf16(y2, oracle.matmul(b(y1.cpu()), b(w2), oracle.W_NK), "chained split-K")
    check_bf16(y3, oracle.matmul(b(y2.cpu()), b(w3), oracle.W_NK), "chained invariant")


def test_matmul_limit_experiment(dev, sms):
    """Rows 0..3 computed alone (M = 1) against the same rows inside M = 2, 4, 8 and 256
    (14 comparisons):
    at limit 0 the M = 256 call runs one K loop per tile while M = 1 splits K, so rows
    differ; with the limit covering 256 every call is the invariant kernel."""
    N, K = 2048, 4096
    gi = inputs.gemm_inputs(256, N, K, seed=11)
    x, w = gi.x.to(dev), gi.w_nk.to(dev)

    def mismatched_rows():
        alone = [bi.matmul(x[i:i + 1], w) for i in range(4)]
        bad = 0
        for M in (2, 4, 8, 256):
            y = bi.matmul(x[:M], w)
            bad += sum(not bits_equal(y[i:i + 1], alone[i]) for i in range(min(4, M)))
        return bad

    bi.set_batch_invariant_limit(0)
    assert bi.matmul_splits(1, N, K, "nk", sms) == 2 and bi.matmul_splits(256, N, K, "nk", sms) == 1
    off = mismatched_rows()
    bi.set_batch_invariant_limit(256)
    on = mismatched_rows()
    assert on == 0
    assert off >= 4, f"limit 0: only {off} of 14 rows differ"


# ------------------------------------------------------------- chosen chunk length

def _to_dev(p, dev):
    return dataclasses.replace(p, **{f.name: getattr(p, f.name).to(dev)
                                     for f in dataclasses.fields(p)
                                     if isinstance(getattr(p, f.name), torch.Tensor)})


FAST_ATTN = [
    # (seq_lens, q_lens, workspace factor over the invariant size)
    ([1028], [8], 8),
    ([65, 400, 1100], [1, 4, 8], 8),
    ([5000, 70, 300], [8, 1, 3], 1),
    ([700] * 24, [2] * 24, 8),
    ([1028] * 8, [8] * 8, 1),
]


@pytest.mark.parametrize("case", range(len(FAST_ATTN)))
def test_chosen_chunk_parity(dev, sms, case):
    bi.set_batch_invariant_limit(0)
    seq_lens, q_lens, factor = FAST_ATTN[case]
    p = inputs.paged_inputs(seq_lens, q_lens, Hq=32, Hkv=8, D=128, seed=300 + case)
    d = _to_dev(p, dev)
    bi.kv_append(d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q)
    T, L, mq = p.T, max(seq_lens), max(q_lens)
    need = factor * bi.attn_workspace_size(T, 32, 128, L)
    c = bi.attn_chunk(len(seq_lens), T, mq, L, 32, 8, 128, need, sms)
    assert c != bi.ATTN_CHUNK, "case does not exercise a non-invariant chunk length"
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out, lse = bi.verify_block(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q,
                               max_q=mq, max_seq_len=L, scale=1.0 / np.sqrt(128), workspace=ws)
    b = inputs.bf16_bits
    kc, vc = b(d.k_cache.cpu()), b(d.v_cache.cpu())
    ref, ref_lse = oracle.attention(b(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                                    p.cu_q.numpy(), 32, 1.0 / np.sqrt(128))
    check_bf16(out, ref, f"chunk {c} case {case}")
    check_rows_rel_l2(out, ref, what=f"chunk {c} case {case}")
    assert np.allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-4)
    # same bits on a repeat
    out2, lse2 = bi.verify_block(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q,
                                 max_q=mq, max_seq_len=L, scale=1.0 / np.sqrt(128), workspace=ws)
    assert bits_equal(out2, out) and bits_equal(lse2, lse)


def test_long_chunks_sampled_parity_and_decode(dev, sms):
    """Eight 65,540-key sequences, one new token each: 2,048-key chunks at limit 0."""
    bi.set_batch_invariant_limit(0)
    L, B = 65540, 8
    p = inputs.paged_inputs([L] * B, [1] * B, Hq=32, Hkv=8, D=128, seed=310, device=dev)
    d = _to_dev(p, dev)
    bi.kv_append(d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q)
    assert bi.attn_chunk(B, B, 1, L, 32, 8, 128, bi.attn_workspace_size(B, 32, 128, L), sms) == 2048
    out, lse = bi.verify_block(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q,
                               max_q=1, max_seq_len=L, scale=1.0 / np.sqrt(128))
    dec, dlse = bi.decode_attn(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens,
                               max_seq_len=L, scale=1.0 / np.sqrt(128))
    assert bits_equal(dec, out) and bits_equal(dlse, lse)
    b = inputs.bf16_bits
    kc, vc = b(d.k_cache.cpu()), b(d.v_cache.cpu())
    for bb, h in ((0, 0), (3, 17), (7, 31)):
        ref, ref_lse = oracle.attention_row(b(p.q.cpu()), kc, vc, p.block_table.cpu().numpy(),
                                            p.seq_lens.cpu().numpy(), p.cu_q.cpu().numpy(),
                                            bb, 0, h, 32, 1.0 / np.sqrt(128))
        check_bf16(out[bb, h], ref, f"2048-key chunks b={bb} h={h}")
        check_rows_rel_l2(out[bb, h], ref, what=f"2048-key chunks b={bb} h={h}")
        assert abs(float(lse[bb, h]) - ref_lse) < 1e-4


@pytest.mark.parametrize("L", [1028, 8196, 16388, 65540])
def test_attention_limit_experiment(dev, sms, L):
    """The pages' SDPA experiment at Lk in {1028, 8196, 16388, 65540}: each query of an
    8-token verify block (here in a batch of 8 such blocks) against the same query decoded
    alone.  At limit 0 the two calls pick different chunk lengths from their load and
    rows differ; at limit 8 all 8 x 32 (query, head) rows match bit for bit."""
    B, q, H = 8, 8, 32
    p = inputs.paged_inputs([L] * B, [q] * B, Hq=H, Hkv=8, D=128, seed=320 + L, device=dev)
    d = _to_dev(p, dev)
    bi.kv_append(d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q)
    scale = 1.0 / np.sqrt(128)

    def mismatched_rows():
        blk, _ = bi.verify_block(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q,
                                 max_q=q, max_seq_len=L, scale=scale)
        bad = 0
        for j in range(q):
            pos = L - q + j
            one, _ = bi.decode_attn(d.q[j:j + 1].contiguous(), d.k_cache, d.v_cache,
                                    d.block_table[:1].contiguous(),
                                    torch.tensor([pos + 1], dtype=torch.int32, device=dev),
                                    max_seq_len=pos + 1, scale=scale)
            bad += int((one[0].view(torch.int16) != blk[j].view(torch.int16)).any(dim=1).sum())
        return bad

    bi.set_batch_invariant_limit(0)
    ws_blk = bi.attn_workspace_size(B * q, H, 128, L)
    c_blk = bi.attn_chunk(B, B * q, q, L, H, 8, 128, ws_blk, sms)
    c_one = bi.attn_chunk(1, 1, 1, L, H, 8, 128, bi.attn_workspace_size(1, H, 128, L), sms)
    assert c_blk != c_one
    off = mismatched_rows()
    bi.set_batch_invariant_limit(8)
    on = mismatched_rows()
    assert on == 0
    assert off > 0, f"L={L}: chunks {c_one} vs {c_blk} but no row differs"
