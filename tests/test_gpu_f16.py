"""IEEE binary16 inputs for bi_matmul_ex and bi_rmsnorm_ex on the GPU: parity with the
oracle (binary16 widened from the format definition, fp32 accumulation), exact integer
cases bit for bit, and batch invariance GPU vs GPU ("Fix/speculative shape invariance",
ml-explore/mlx PR 4279, the tester's comment: dense matmul divergence shows for f16
inputs too)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_f16, check_f32

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _half_inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g).to(torch.float16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.float16)
    return x, w


def _scale(x, w):
    return np.abs(x.float().numpy().astype(np.float64)) @ np.abs(w.float().numpy().astype(np.float64)).T


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (8, 4096, 4096), (3, 200, 200), (130, 96, 320),
                                   (1800, 4000, 328)])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_f16_matmul_matches_oracle(dev, M, N, K, layout):
    if layout == "kn" and N % 8:
        pytest.skip("KN layout needs N % 8 == 0")
    x, w = _half_inputs(M, N, K, M + N + K)
    wl = w if layout == "nk" else w.t().contiguous()
    rows = list(range(M)) if M <= 130 else [0, 127, 128, 255, 256, 1024, M - 1]
    ref = oracle.matmul16(_bits(x[rows]), _bits(w), oracle.W_NK, oracle.F16)
    scale = _scale(x[rows], w)
    y = bi.matmul(x.to(dev), wl.to(dev), layout).cpu()
    assert y.dtype == torch.float16
    check_f16(y[rows], ref, scale, f"f16 matmul {layout} {M}x{N}x{K}")
    y32 = bi.matmul(x.to(dev), wl.to(dev), layout, out_dtype=torch.float32).cpu()
    check_f32(y32[rows], ref, scale, f"f16 matmul fp32 out {layout} {M}x{N}x{K}")


def test_f16_matmul_exact_integers_bit_exact(dev):
    M, N, K = 40, 96, 1024
    x = inputs.small_int_bf16((M, K), -8, 8, 0, seed=31).float().to(torch.float16)
    w = inputs.small_int_bf16((N, K), -8, 8, -4, seed=32).float().to(torch.float16)
    y = bi.matmul(x.to(dev), w.to(dev), "nk", out_dtype=torch.float32).cpu().numpy()
    assert np.array_equal(y, oracle.matmul16(_bits(x), _bits(w), oracle.W_NK, oracle.F16))


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_f16_matmul_rows_invariant_across_M(dev, layout):
    K = N = 4096
    x, w = _half_inputs(2048, N, K, 5)
    wl = (w if layout == "nk" else w.t().contiguous()).to(dev)
    xd = x.to(dev)
    full = bi.matmul(xd, wl, layout)
    for M in (1, 2, 4, 8, 9, 64, 128, 129, 1000, 1500):
        assert bits_equal(bi.matmul(xd[:M].contiguous(), wl, layout), full[:M]), M


@pytest.mark.parametrize("rows,H", [(1, 256), (4, 4096), (2048, 4096), (3, 20000)])
def test_f16_rmsnorm_matches_oracle_and_is_invariant(dev, rows, H):
    g = torch.Generator().manual_seed(rows + H)
    x = (torch.randn(rows, H, generator=g) * 3).to(torch.float16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.float16)
    ref = oracle.rmsnorm16(_bits(x), _bits(gamma), 1e-5, oracle.F16)
    y = bi.rmsnorm(x.to(dev), gamma.to(dev), 1e-5)
    assert y.dtype == torch.float16
    check_f16(y.cpu(), ref, np.abs(ref), f"f16 rmsnorm {rows}x{H}")
    for i in (0, rows - 1):
        alone = bi.rmsnorm(x[i:i + 1].to(dev), gamma.to(dev), 1e-5)
        assert bits_equal(alone, y[i:i + 1])
