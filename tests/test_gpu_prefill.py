"""bi_prefill_attn on the GPU: chunked prefill and prefix caching (book chapter
"Batch-invariant kernels: why temperature-0 decoding is still nondeterministic", Case 6 and
the paragraph after its strategy table: serving engines slice sequences, and token 1000
must reduce identically whether 0 or 999 tokens are already cached; the cache and the new
tokens are scored in one loop).

Parity with the CPU oracle, and bit-identity of every query across the ways of reaching
it: the whole prompt in one call, the prompt cut into chunks of assorted sizes, verify
blocks of up to 8 tokens, single-token decoding, and other sequences in the same call."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16, check_rows_rel_l2

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to_dev(p, dev):
    return dataclasses.replace(p, **{f.name: getattr(p, f.name).to(dev)
                                     for f in dataclasses.fields(p)
                                     if isinstance(getattr(p, f.name), torch.Tensor)})


def _appended(p, dev):
    d = _to_dev(p, dev)
    bi.kv_append(d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q)
    return d


def _prefill(d, q, bt, sl, cu, D):
    mq = int((cu[1:] - cu[:-1]).max())
    return bi.prefill_attn(q, d.k_cache, d.v_cache, bt, sl, cu, max_q=mq,
                           max_seq_len=int(sl.max()), scale=1.0 / np.sqrt(D))


def _i32(x, dev):
    return torch.tensor(x, dtype=torch.int32, device=dev)


CASES = [
    # (seq_lens, q_lens, Hq, Hkv, D): the block is the last q_len tokens of each sequence
    ([300], [300], 8, 2, 128),                  # a whole prompt, G = 4: 32 tokens per tile
    ([1100, 700], [600, 700], 8, 2, 128),       # 500 cached + 600 new; a fresh 700
    ([520, 64, 1], [520, 64, 1], 4, 4, 64),     # G = 1: 128 tokens per tile, head_dim 64
    ([900], [200], 16, 2, 128),                 # G = 8: 16 tokens per tile
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_parity(dev, case):
    lens, qls, Hq, Hkv, D = CASES[case]
    p = inputs.paged_inputs(lens, qls, Hq=Hq, Hkv=Hkv, D=D, seed=100 + case)
    d = _appended(p, dev)
    out, lse = _prefill(d, d.q, d.block_table, d.seq_lens, d.cu_q, D)
    b16 = inputs.bf16_bits
    kc, vc = oracle.kv_append(b16(p.k_new), b16(p.v_new), b16(p.k_cache), b16(p.v_cache),
                              p.block_table.numpy(), p.seq_lens.numpy(), p.cu_q.numpy(), 64)
    ref, ref_lse = oracle.attention(b16(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                                    p.cu_q.numpy(), Hq, 1.0 / np.sqrt(D))
    check_bf16(out, ref, f"prefill case {case}")
    check_rows_rel_l2(out, ref, what=f"prefill case {case}")
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < 1e-4


def test_prefill_chunks_verify_and_decode_agree_bitwise(dev):
    """One prompt of 1,100 tokens (chunks of 512 keys: 0, 1, 2): the whole prompt in one
    call, then cut into chunks of 100 / 333 / 207 / 460 tokens (each chunk after the ones
    before it are cached), verify blocks of 8 across the chunk boundaries, and single
    tokens decoded alone: every query's out and lse bits are the same."""
    L, Hq, Hkv, D = 1100, 32, 8, 128
    p = inputs.paged_inputs([L], [L], Hq=Hq, Hkv=Hkv, D=D, seed=7)
    d = _appended(p, dev)
    bt = d.block_table
    full, full_lse = _prefill(d, d.q, bt, d.seq_lens, d.cu_q, D)
    cuts = [0, 100, 433, 640, 1100]
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = _prefill(d, d.q[a:b].contiguous(), bt, _i32([b], dev), _i32([0, b - a], dev), D)
        assert bits_equal(o, full[a:b]) and bits_equal(l, full_lse[a:b]), f"chunk {a}:{b}"
    for a in (0, 504, 508, 1016, 1092):
        b = a + 8
        o, l = bi.verify_block(d.q[a:b].contiguous(), d.k_cache, d.v_cache, bt, _i32([b], dev),
                               _i32([0, 8], dev), max_q=8, max_seq_len=b, scale=1.0 / np.sqrt(D))
        assert bits_equal(o, full[a:b]) and bits_equal(l, full_lse[a:b]), f"verify {a}:{b}"
    for t in (0, 1, 63, 64, 511, 512, 513, 1023, 1024, 1099):
        o, l = bi.decode_attn(d.q[t:t + 1].contiguous(), d.k_cache, d.v_cache, bt,
                              _i32([t + 1], dev), max_seq_len=t + 1, scale=1.0 / np.sqrt(D))
        assert bits_equal(o, full[t:t + 1]) and bits_equal(l, full_lse[t:t + 1]), f"decode {t}"
        o2, l2 = _prefill(d, d.q[t:t + 1].contiguous(), bt, _i32([t + 1], dev),
                          _i32([0, 1], dev), D)
        assert bits_equal(o2, o) and bits_equal(l2, l), f"one-token prefill {t}"


def test_prefill_mixed_batch_equals_each_sequence_alone(dev):
    """Sequences of mixed lengths and block widths in one call (tiles, chunks and heads of
    different sequences spread over the CTAs) give each sequence's bits alone."""
    lens = [1300, 70, 513, 2049, 5]
    qls = [1300, 33, 200, 129, 5]
    p = inputs.paged_inputs(lens, qls, Hq=16, Hkv=4, D=128, seed=21)
    d = _appended(p, dev)
    out, lse = _prefill(d, d.q, d.block_table, d.seq_lens, d.cu_q, 128)
    for b in range(len(lens)):
        c0, c1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        o, l = _prefill(d, d.q[c0:c1].contiguous(), d.block_table[b:b + 1].contiguous(),
                        d.seq_lens[b:b + 1].contiguous(), _i32([0, c1 - c0], dev), 128)
        assert bits_equal(o, out[c0:c1]) and bits_equal(l, lse[c0:c1]), f"sequence {b}"
    # sampled rows against the oracle
    b16 = inputs.bf16_bits
    kc, vc = b16(d.k_cache.cpu()), b16(d.v_cache.cpu())
    for b, j, h in ((0, 0, 0), (0, 1299, 15), (3, 128, 7), (4, 4, 3)):
        ref, ref_lse = oracle.attention_row(b16(p.q), kc, vc, p.block_table.numpy(),
                                            p.seq_lens.numpy(), p.cu_q.numpy(), b, j, h, 16,
                                            1.0 / np.sqrt(128))
        t = int(p.cu_q[b]) + j
        check_bf16(out[t, h], ref, f"mixed prefill row b={b} j={j} h={h}")
        check_rows_rel_l2(out[t, h], ref, what=f"mixed prefill row b={b} j={j} h={h}")
        assert abs(float(lse[t, h]) - ref_lse) < 1e-4


def test_prefill_repeat_and_guard_bands(dev):
    """Run-to-run identical; nothing written outside out and lse."""
    p = inputs.paged_inputs([700], [300], Hq=8, Hkv=2, D=128, seed=33)
    d = _appended(p, dev)
    T, Hq, D = p.q.shape
    obuf = torch.full((T + 2, Hq, D), 3.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((T + 2, Hq), 5.0, dtype=torch.float32, device=dev)
    seen = set()
    for _ in range(10):
        bi.prefill_attn(d.q, d.k_cache, d.v_cache, d.block_table, d.seq_lens, d.cu_q,
                        max_q=300, max_seq_len=700, scale=1.0 / np.sqrt(D), out=obuf[1:T + 1],
                        lse=lbuf[1:T + 1])
        seen.add(bytes(obuf[1:T + 1].contiguous().view(torch.int16).cpu().numpy()))
    assert len(seen) == 1
    assert torch.all(obuf[0] == 3.0) and torch.all(obuf[T + 1] == 3.0)
    assert torch.all(lbuf[0] == 5.0) and torch.all(lbuf[T + 1] == 5.0)
    assert bi.device_status() == bi.BI_OK
