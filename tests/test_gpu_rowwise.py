"""bi_log_softmax and bi_mean (include/bi_rowwise.h) on the GPU against the oracle, and
their batch invariance GPU vs GPU, bit for bit: a row alone equals the row in a batch, at
any alignment or stride (book chapter "Batch-invariant kernels...", The boring rule item 2;
Sources: the mean and log-softmax overrides)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_f32

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _logits(rows, n, seed, std=4.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(rows, n, generator=g) * std


# n picks the cut of a row: registers of one CTA (1..16,384), a cluster of 2..8 CTAs with
# 16 (..131,072) or 32 (..262,144) values per thread, or a streamed row beyond
@pytest.mark.parametrize("rows,n", [(1, 1), (3, 5), (8, 4097), (33, 128256), (2, 4099),
                                    (2, 200001), (2, 300000)])
def test_log_softmax_matches_oracle(dev, rows, n):
    x = _logits(rows, n, 500 + n)
    if n > 4:
        x[0, 1] = float("-inf")
        x[-1, :] = x[-1, :] * 100.0          # large magnitudes: the max shift matters
    want = oracle.log_softmax(x.numpy())
    got = bi.log_softmax(x.to(dev))
    g = got.cpu().numpy()
    finite = np.isfinite(want)
    assert np.array_equal(np.isneginf(g), np.isneginf(want))
    # fp32 exp, tree sum and log against the fp64 definition
    check_f32(got.cpu()[torch.from_numpy(finite)], want[finite], 1.0 + np.abs(want[finite]),
              f"log_softmax {rows}x{n}")


def test_log_softmax_special_rows(dev):
    x = torch.zeros(4, 6)
    x[0, 2] = float("nan")
    x[1, :] = float("-inf")
    x[2, 3] = float("inf")
    got = bi.log_softmax(x.to(dev)).cpu()
    assert torch.isnan(got[:3]).all()
    assert torch.allclose(got[3], torch.full((6,), -float(np.log(6.0))))


def test_log_softmax_rows_invariant_alignment_and_in_place(dev):
    n = 50257
    x = _logits(16, n, 7).to(dev)
    full = bi.log_softmax(x)
    for i in (0, 5, 15):
        assert bits_equal(bi.log_softmax(x[i:i + 1].contiguous()), full[i:i + 1])
    # the same rows at an odd offset and stride (scalar loads instead of 128-bit ones)
    big = torch.empty(16 * (n + 3) + 1, device=dev)
    strided = big[1:1 + 16 * (n + 3)].view(16, n + 3)[:, :n]
    strided.copy_(x)
    out = torch.empty_like(strided)
    assert bits_equal(bi.log_softmax(strided, out=out), full)
    # in place
    y = x.clone()
    bi.log_softmax(y, out=y)
    assert bits_equal(y, full)
    seen = {bytes(bi.log_softmax(x).cpu().numpy()) for _ in range(20)}
    assert len(seen) == 1


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,n", [(1, 1), (7, 3), (64, 4096), (5, 50257), (2, 200001),
                                    (3, 1000003)])
def test_mean_matches_oracle(dev, dtype, rows, n):
    x = _logits(rows, n, 600 + n, std=2.0) + 0.5
    xd = x.to(dtype)
    if dtype == torch.bfloat16:
        want = oracle.mean(inputs.bf16_bits(xd), bf16=True)
    else:
        want = oracle.mean(x.numpy())
    got = bi.mean(xd.to(dev))
    scale = np.abs(xd.float().numpy()).mean(axis=1)
    check_f32(got, want, scale, f"mean {dtype} {rows}x{n}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mean_rows_invariant(dev, dtype):
    n = 4099
    x = _logits(32, n, 9).to(dtype).to(dev)
    full = bi.mean(x)
    for i in (0, 31):
        assert bits_equal(bi.mean(x[i:i + 1].contiguous()), full[i:i + 1])
    big = torch.empty(32 * (n + 1) + 1, dtype=dtype, device=dev)
    strided = big[1:1 + 32 * (n + 1)].view(32, n + 1)[:, :n]
    strided.copy_(x)
    assert bits_equal(bi.mean(strided), full)
