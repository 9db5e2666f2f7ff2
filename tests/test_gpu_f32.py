"""fp32 inputs for bi_matmul_ex and bi_rmsnorm_ex on the GPU ("Fix/speculative shape
invariance", ml-explore/mlx PR 4279, the tester's comment: f32 dense matmul diverges
with the limit off): parity with the oracle, exact integers bit for bit, and rows
bitwise across M / batch (GPU vs GPU)."""
import numpy as np
import pytest
import torch

import oracle
from tolerance import bits_equal, check_f32

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(M, K, generator=g), torch.randn(N, K, generator=g) * 0.02


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (4, 4096, 4096), (3, 200, 203), (130, 96, 320),
                                   (17, 1000, 37)])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_f32_matmul_matches_oracle(dev, M, N, K, layout):
    x, w = _inputs(M, N, K, M * 3 + N + K)
    wl = w if layout == "nk" else w.t().contiguous()
    y = bi.matmul(x.to(dev), wl.to(dev), layout)
    ref = oracle.matmul_f32(x.numpy(), w.numpy(), oracle.W_NK)
    scale = np.abs(x.numpy().astype(np.float64)) @ np.abs(w.numpy().astype(np.float64)).T
    check_f32(y, ref, scale, f"f32 matmul {layout} {M}x{N}x{K}")


def test_f32_matmul_exact_integers(dev):
    g = torch.Generator().manual_seed(8)
    x = torch.randint(-64, 65, (20, 300), generator=g).float()
    w = torch.randint(-64, 65, (33, 300), generator=g).float()
    y = bi.matmul(x.to(dev), w.to(dev), "nk").cpu().numpy()
    assert np.array_equal(y, oracle.matmul_f32(x.numpy(), w.numpy(), oracle.W_NK))


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_f32_matmul_rows_invariant_across_M(dev, layout):
    N, K = 1024, 1000
    x, w = _inputs(300, N, K, 9)
    wl = (w if layout == "nk" else w.t().contiguous()).to(dev)
    xd = x.to(dev)
    full = bi.matmul(xd, wl, layout)
    for M in (1, 2, 4, 8, 16, 17, 64, 65, 299):
        assert bits_equal(bi.matmul(xd[:M].contiguous(), wl, layout), full[:M]), M
    # the limit has no effect on the fp32 path
    old = bi.get_batch_invariant_limit()
    bi.set_batch_invariant_limit(0)
    try:
        assert bits_equal(bi.matmul(xd[:4].contiguous(), wl, layout), full[:4])
    finally:
        bi.set_batch_invariant_limit(old)


@pytest.mark.parametrize("rows,H", [(1, 1), (5, 4096), (300, 8192), (2, 20001)])
def test_f32_rmsnorm_matches_oracle_and_is_invariant(dev, rows, H):
    g = torch.Generator().manual_seed(rows + H)
    x = torch.randn(rows, H, generator=g) * 3
    gamma = 1 + 0.1 * torch.randn(H, generator=g)
    ref = oracle.rmsnorm_f32(x.numpy(), gamma.numpy(), 1e-5)
    y = bi.rmsnorm(x.to(dev), gamma.to(dev), 1e-5)
    check_f32(y, ref, np.abs(ref) + 1e-30, f"f32 rmsnorm {rows}x{H}")
    for i in (0, rows - 1):
        assert bits_equal(bi.rmsnorm(x[i:i + 1].to(dev), gamma.to(dev), 1e-5), y[i:i + 1])
