"""bi_rmsnorm on the GPU: parity with the CPU oracle, closed forms, batch invariance.

Book chapter "Batch-invariant kernels...", Case 4 and Case 6 (RMSNorm row): a row's
bits must be the same served alone or inside any batch.
"""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16, check_f32

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.mark.parametrize("B,H,eps", [(1, 256, 1e-6), (8, 256, 1e-6), (3, 8192, 1e-5),
                                     (16, 4096, 1e-5), (5, 1001, 1e-5), (2, 7, 0.1),
                                     (4, 20000, 1e-5), (33, 2056, 1e-6)])
def test_rmsnorm_parity(dev, B, H, eps):
    x, gamma = inputs.rmsnorm_inputs(B, H, seed=B * 31 + H)
    y = bi.rmsnorm(x.to(dev), gamma.to(dev), eps)
    ref = oracle.rmsnorm(inputs.bf16_bits(x), inputs.bf16_bits(gamma), eps)
    check_bf16(y, ref, f"rmsnorm {B}x{H}")
    yf = bi.rmsnorm(x.to(dev), gamma.to(dev), eps, out_dtype=torch.float32)
    check_f32(yf, ref, np.abs(ref), f"rmsnorm f32 {B}x{H}")


def test_rmsnorm_rows_invariant_across_batch(dev):
    """The pages' RMSNorm workload: hidden 8192, B in {1,3,16,128,2048}, outliers x50."""
    x, gamma = inputs.rmsnorm_inputs(2048, 8192, seed=3)
    x, gamma = x.to(dev), gamma.to(dev)
    full = bi.rmsnorm(x, gamma, 1e-5)
    for B in (1, 3, 16, 128):
        assert bits_equal(bi.rmsnorm(x[:B].contiguous(), gamma, 1e-5), full[:B])
    for i in (7, 1000, 2047):
        assert bits_equal(bi.rmsnorm(x[i:i + 1].contiguous(), gamma, 1e-5), full[i:i + 1])
    perm = torch.randperm(2048, generator=inputs.generator(5)).to(dev)
    assert bits_equal(bi.rmsnorm(x[perm].contiguous(), gamma, 1e-5), full[perm])
    # sampled parity at full size
    ref_rows = oracle.rmsnorm(inputs.bf16_bits(x[[0, 1, 2047]].cpu()),
                              inputs.bf16_bits(gamma.cpu()), 1e-5)
    check_bf16(full[[0, 1, 2047]], ref_rows, "rmsnorm full-size sample")


def test_rmsnorm_alignment_paths_same_bits(dev):
    """A row read through unaligned (scalar) loads gives the bits of the aligned path."""
    x, gamma = inputs.rmsnorm_inputs(6, 4096, seed=9)
    xd, gd = x.to(dev), gamma.to(dev)
    aligned = bi.rmsnorm(xd, gd, 1e-5)
    buf = torch.zeros(6, 4096 + 3, dtype=torch.bfloat16, device=dev)
    buf[:, 3:] = xd
    shifted = bi.rmsnorm(buf[:, 3:], gd, 1e-5)
    assert bits_equal(shifted, aligned)


def test_rmsnorm_closed_forms(dev):
    H = 4096
    g = inputs.generator(6)
    signs = torch.where(torch.rand(H, generator=g) < 0.5, -1.0, 1.0)
    x = (signs * 8.0).to(torch.bfloat16)[None]
    gamma = torch.ones(H, dtype=torch.bfloat16)
    y = bi.rmsnorm(x.to(dev), gamma.to(dev), 0.0, out_dtype=torch.float32).cpu()
    # rsqrt(64) within its error bound of 1/8: y = +-1 within a few ulp
    assert torch.allclose(y[0], signs, rtol=4e-7, atol=0)
    # book chapter Case 4 row: the GPU sum of squares matches the closed form
    row = torch.tensor([2.0 ** -(i // 64) for i in range(H)], dtype=torch.float32)
    yr = bi.rmsnorm(row.to(torch.bfloat16)[None].to(dev), gamma.to(dev), 0.0,
                    out_dtype=torch.float32).cpu()[0]
    ss_closed = (256.0 / 3.0) * (1 - 4.0 ** -64)
    inv = 1 / np.sqrt(ss_closed / H)
    assert np.allclose(yr.numpy(), row.numpy() * inv, rtol=2e-6, atol=0)


def test_rmsnorm_guard_bands_and_errors(dev):
    x, gamma = inputs.rmsnorm_inputs(3, 100, seed=11)
    buf = torch.full((5, 128), 9.0, dtype=torch.float32, device=dev)
    bi.rmsnorm(x.to(dev), gamma.to(dev), 1e-5, out=buf[1:4, 4:104])
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask[1:4, 4:104] = False
    assert torch.all(buf[mask] == 9.0)
    with pytest.raises(bi.BIError) as e:
        bi.rmsnorm(x.to(dev), gamma.to(dev), -1.0)
    assert e.value.status == bi.BI_ERR_INVALID_ARG
    bi.rmsnorm(x[:0].to(dev), gamma.to(dev), 1e-5)   # rows = 0: no-op
    assert bi.device_status() == bi.BI_OK


def test_rmsnorm_repeat_runs_one_result(dev):
    x, gamma = inputs.rmsnorm_inputs(64, 8192, seed=13)
    xd, gd = x.to(dev), gamma.to(dev)
    outs = {bytes(bi.rmsnorm(xd, gd, 1e-5).view(torch.int16).cpu().numpy()) for _ in range(100)}
    assert len(outs) == 1
