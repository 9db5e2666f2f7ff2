"""Decoder glue on the GPU (include/bi_glue.h) against the oracle: embedding gather and
argmax bit-exact, residual add bit-exact where the fp32 sum is exact, rotary embedding
and SwiGLU within the bf16 tolerance of the unrounded fp64 oracle; a token's rotary
embedding alone equals the same token inside a ragged block, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _bits(t):
    return inputs.bf16_bits(t)


# ------------------------------------------------------------------------ embedding

def test_embedding_gathers_rows_exactly(dev):
    table = inputs.normal_bf16((1000, 256), std=0.02, seed=401).to(dev)
    ids = torch.tensor([0, 999, 5, 5, 123, 0, 777], dtype=torch.int32, device=dev)
    out = bi.embedding(table, ids)
    assert bits_equal(out, table[ids.long()])
    assert bi.device_status() == bi.BI_OK


def test_embedding_out_of_range_id_writes_zeros_and_reports(dev):
    table = inputs.normal_bf16((100, 64), seed=402).to(dev)
    ids = torch.tensor([3, 100, -1, 7], dtype=torch.int32, device=dev)
    out = torch.full((4, 64), 7.0, dtype=torch.bfloat16, device=dev)
    bi.embedding(table, ids, out=out)
    assert bi.device_status() == bi.BI_ERR_DEVICE_ARG
    assert bits_equal(out[[0, 3]], table[[3, 7]])
    assert torch.all(out[1:3] == 0)
    assert bi.device_status() == bi.BI_OK  # the word was cleared


# ----------------------------------------------------------------------------- RoPE

ROPE_CASES = [  # (seq_lens, q_lens, H, D, theta)
    ([1], [1], 4, 64, 10000.0),
    ([5, 3, 8448], [2, 1, 4], 32, 128, 500000.0),
    ([65540, 700], [8, 3], 8, 128, 500000.0),
    ([17] * 9, [1] * 9, 2, 64, 500000.0),
    ([40], [8], 3, 16, 10000.0),
]


@pytest.mark.parametrize("seq_lens,q_lens,H,D,theta", ROPE_CASES)
def test_rope_matches_oracle(dev, seq_lens, q_lens, H, D, theta):
    T = sum(q_lens)
    x = inputs.normal_bf16((T, H, D), std=2.0, seed=403 + T)
    sl = torch.tensor(seq_lens, dtype=torch.int32)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    want = oracle.rope(_bits(x), oracle.positions(sl.numpy(), cu.numpy()), theta)
    xd = x.to(dev)
    bi.rope(xd, sl.to(dev), cu.to(dev), theta)
    check_bf16(xd, want, "rope vs oracle")
    assert bi.device_status() == bi.BI_OK


def test_rope_decode_form_and_strided_rows(dev):
    # q of a fused [T, (Hq + 2 Hkv) * D] projection: rotate only the first Hq heads
    B, Hq, D = 5, 4, 128
    fused = inputs.normal_bf16((B, (Hq + 4) * D), seed=404)
    sl = torch.tensor([9, 100, 1, 8448, 33], dtype=torch.int32)
    want = oracle.rope(_bits(fused[:, :Hq * D].reshape(B, Hq, D)), oracle.positions(sl.numpy()),
                       500000.0)
    fd = fused.to(dev)
    q = fd[:, :Hq * D].view(B, Hq, D)
    bi.rope(q, sl.to(dev), None, 500000.0)
    check_bf16(q, want, "strided decode rope vs oracle")
    assert bits_equal(fd[:, Hq * D:], fused[:, Hq * D:].to(dev))  # the rest untouched


def test_rope_token_alone_equals_token_in_block(dev):
    H, D, L = 8, 128, 8196
    x = inputs.normal_bf16((4, H, D), seed=405).to(dev)
    block = x.clone()
    bi.rope(block, torch.tensor([L], dtype=torch.int32, device=dev),
            torch.tensor([0, 4], dtype=torch.int32, device=dev))
    for j in range(4):
        alone = x[j:j + 1].clone()
        bi.rope(alone, torch.tensor([L - 4 + j + 1], dtype=torch.int32, device=dev), None)
        assert bits_equal(alone[0], block[j])


def test_rope_bad_block_reports_and_leaves_tokens(dev):
    x = inputs.normal_bf16((3, 2, 64), seed=406).to(dev)
    before = x.clone()
    # sequence 0 claims 3 tokens but holds only 2
    bi.rope(x, torch.tensor([2], dtype=torch.int32, device=dev),
            torch.tensor([0, 3], dtype=torch.int32, device=dev))
    assert bi.device_status() == bi.BI_ERR_DEVICE_ARG
    assert bits_equal(x, before)


# --------------------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("rows,inter", [(1, 8), (3, 512), (32, 14336), (128, 1000)])
def test_swiglu_matches_oracle(dev, rows, inter):
    g = inputs.normal_bf16((rows, inter), std=3.0, seed=407 + rows)
    u = inputs.normal_bf16((rows, inter), std=1.0, seed=408 + rows)
    want = oracle.swiglu(_bits(g), _bits(u))
    out = bi.swiglu(g.to(dev), u.to(dev))
    check_bf16(out, want, "swiglu vs oracle")


def test_swiglu_strided_halves_of_a_fused_projection(dev):
    rows, inter = 6, 256
    gu = inputs.normal_bf16((rows, 2 * inter), std=2.0, seed=409)
    want = oracle.swiglu(_bits(gu[:, :inter]), _bits(gu[:, inter:]))
    d = gu.to(dev)
    out = bi.swiglu(d[:, :inter], d[:, inter:])
    check_bf16(out, want, "strided swiglu vs oracle")


# ------------------------------------------------------------------------------ add

@pytest.mark.parametrize("n", [1, 7, 8, 4096, 4096 * 33 + 5])
def test_add_matches_oracle_bitwise(dev, n):
    # N(0,1) + N(0,1) in bf16: the fp32 sum is exact, so one rounding on each side
    a = inputs.normal_bf16((n,), seed=410 + n)
    b = inputs.normal_bf16((n,), seed=411 + n)
    want = oracle.to_bf16(oracle.add(_bits(a), _bits(b)))
    got = bi.add(a.to(dev), b.to(dev))
    assert np.array_equal(_bits(got.cpu()), want)


def test_add_in_place(dev):
    a = inputs.normal_bf16((1000,), seed=412).to(dev)
    b = inputs.normal_bf16((1000,), seed=413).to(dev)
    want = bi.add(a, b)
    bi.add(a, b, out=a)
    assert bits_equal(a, want)


# --------------------------------------------------------------------------- argmax

def _argmax_rows(dev, n, rows, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, n, generator=g)
    return x


@pytest.mark.parametrize("rows,n", [(1, 1), (3, 5), (8, 4097), (33, 128256)])
def test_argmax_matches_oracle(dev, rows, n):
    x = _argmax_rows(dev, n, rows, 414 + n)
    if n > 4:
        x[0, n // 3] = x[0, n - 2] = 1e9        # a tie: the lower index wins
        if rows > 1:
            x[1, :] = float("nan")              # all NaN: index 0
        if rows > 2:
            x[2, ::2] = float("nan")            # NaN ranks below numbers
            x[2, 1] = float("-inf")
    want = [oracle.argmax_f32(r) for r in x.numpy()]
    got = bi.argmax(x.to(dev)).cpu().tolist()
    assert got == want


def test_argmax_strided_rows(dev):
    x = _argmax_rows(dev, 1003, 4, 415)
    big = torch.zeros(4, 1008)
    big[:, :1003] = x
    big[:, 1003:] = 1e30                         # beyond n: must be ignored
    got = bi.argmax(big.to(dev)[:, :1003]).cpu().tolist()
    assert got == [oracle.argmax_f32(r) for r in x.numpy()]
