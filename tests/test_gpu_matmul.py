"""bi_matmul on the GPU: parity with the CPU oracle, exact cases, batch invariance.

Invariance is judged GPU vs GPU, bit for bit: row i of Y must be identical at every M
(book chapter "Batch-invariant kernels...", "The boring rule" item 2: f(x[None]) vs
f(batch)[0] across batch sizes), under a batch permutation (Try-this item 1), and over
repeated runs.
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


def _abs_scale(x, w_nk):
    X = np.abs(x.float().numpy().astype(np.float64))
    W = np.abs(w_nk.float().numpy().astype(np.float64))
    return X @ W.T


SHAPES = [
    (1, 256, 256), (4, 256, 256), (8, 256, 256),       # tiny single-layer check
    (3, 200, 200),                                     # ragged N and K tails
    (130, 96, 320),                                    # two M tiles, ragged M
    (257, 64, 64), (5, 33, 8), (2, 1000, 1032),
    (61, 304, 520),                                    # M = 64 instructions, every lane quarter
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_parity_bf16(dev, M, N, K, layout):
    if layout == "kn" and N % 8 != 0:
        pytest.skip("KN layout needs N % 8 == 0 for the TMA row stride")
    gi = inputs.gemm_inputs(M, N, K, seed=M * 7 + N + K)
    w = gi.w_nk if layout == "nk" else gi.w_kn
    y = bi.matmul(gi.x.to(dev), w.to(dev), layout)
    ref = oracle.matmul(inputs.bf16_bits(gi.x), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_bf16(y, ref, f"matmul {layout} {M}x{N}x{K}")


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_parity_f32(dev, layout):
    M, N, K = 9, 160, 704
    gi = inputs.gemm_inputs(M, N, K, seed=21)
    w = gi.w_nk if layout == "nk" else gi.w_kn
    y = bi.matmul(gi.x.to(dev), w.to(dev), layout, out_dtype=torch.float32)
    ref = oracle.matmul(inputs.bf16_bits(gi.x), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_f32(y, ref, _abs_scale(gi.x, gi.w_nk), f"matmul f32 {layout}")


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_exact_integers_bit_exact(dev, layout):
    """Integer-valued operands: every order is exact, so GPU == oracle bit for bit."""
    M, N, K = 40, 96, 1024
    x = inputs.small_int_bf16((M, K), -8, 8, 0, seed=31)
    w_nk = inputs.small_int_bf16((N, K), -8, 8, -4, seed=32)
    w = w_nk if layout == "nk" else w_nk.t().contiguous()
    y = bi.matmul(x.to(dev), w.to(dev), layout, out_dtype=torch.float32)
    ref = oracle.matmul(inputs.bf16_bits(x), inputs.bf16_bits(w_nk), oracle.W_NK)
    assert np.array_equal(y.cpu().numpy(), ref)
    yb = bi.matmul(x.to(dev), w.to(dev), layout)
    assert np.array_equal(inputs.bf16_bits(yb.cpu()), oracle.bf16_round(ref))


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_rows_invariant_across_M(dev, layout):
    """The pages' GEMM workload: K=N=4096, M in {1,...,2048}; row i identical at every M."""
    K = N = 4096
    gi = inputs.gemm_inputs(2048, N, K, seed=2)
    w = (gi.w_nk if layout == "nk" else gi.w_kn).to(dev)
    x = gi.x.to(dev)
    full = bi.matmul(x, w, layout)
    # every M crosses a different staging / CTA-tiling choice of the scheduler:
    # staged X rows 8..128, one to eight 32-wide instruction tiles per CTA, M = 64
    # instructions up to 64 rows (rows in all four lane quarters from M = 49) and M = 128
    # ones from 65
    for M in (1, 2, 3, 4, 8, 9, 16, 17, 33, 49, 64, 65, 100, 127, 128, 129, 256, 600, 1000,
              1500):
        part = bi.matmul(x[:M].contiguous(), w, layout)
        assert bits_equal(part, full[:M]), f"rows differ at M={M}"
    # a row evaluated alone from the middle of the batch (not only the first rows)
    for i in (5, 127, 128, 1999):
        alone = bi.matmul(x[i:i + 1].contiguous(), w, layout)
        assert bits_equal(alone, full[i:i + 1]), f"row {i} differs alone"


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_full_size_sampled_parity(dev, layout):
    K = N = 4096
    gi = inputs.gemm_inputs(2048, N, K, seed=2)
    w = gi.w_nk if layout == "nk" else gi.w_kn
    y = bi.matmul(gi.x.to(dev), w.to(dev), layout).cpu()
    wb = inputs.bf16_bits(gi.w_nk)
    for i in (0, 127, 128, 1024, 2047):
        ref = oracle.matmul(inputs.bf16_bits(gi.x[i:i + 1]), wb, oracle.W_NK)
        check_bf16(y[i:i + 1], ref, f"row {i}")


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_parity_wide_cta_tiles_ragged_n(dev, layout):
    """Large M (several instruction tiles per CTA) with N not a multiple of the CTA tile."""
    M, N, K = 1500, 1000, 256
    gi = inputs.gemm_inputs(M, N, K, seed=81)
    w = gi.w_nk if layout == "nk" else gi.w_kn
    y = bi.matmul(gi.x.to(dev), w.to(dev), layout).cpu()
    rows = [0, 1, 127, 128, 700, 1499]
    ref = oracle.matmul(inputs.bf16_bits(gi.x[rows]), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_bf16(y[rows], ref, f"wide tiles {layout}")
    yf = bi.matmul(gi.x.to(dev), w.to(dev), layout, out_dtype=torch.float32).cpu()
    check_f32(yf[rows], ref, _abs_scale(gi.x[rows], gi.w_nk), f"wide tiles f32 {layout}")
    # and every row of this launch equals the row computed alone
    for i in (3, 1499):
        alone = bi.matmul(gi.x[i:i + 1].to(dev), w.to(dev), layout).cpu()
        assert bits_equal(alone, y[i:i + 1])


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_matmul_parity_256_row_tiles_ragged(dev, layout):
    """Large M and N: 256 x 256 CTA tiles (two instruction tiles along M), with M, N and
    K all ragged (K not a multiple of the 64-wide K-block)."""
    M, N, K = 1800, 4000, 328
    gi = inputs.gemm_inputs(M, N, K, seed=83)
    w = gi.w_nk if layout == "nk" else gi.w_kn
    y = bi.matmul(gi.x.to(dev), w.to(dev), layout).cpu()
    rows = [0, 127, 128, 255, 256, 1024, 1791, 1799]
    ref = oracle.matmul(inputs.bf16_bits(gi.x[rows]), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_bf16(y[rows], ref, f"256-row tiles {layout}")
    for i in (128, 1799):
        alone = bi.matmul(gi.x[i:i + 1].to(dev), w.to(dev), layout).cpu()
        assert bits_equal(alone, y[i:i + 1])


@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("M,N,K", [(300, 904, 1000), (512, 4096, 4096), (96, 2000, 520)])
def test_matmul_mid_m_ragged_guard_bands(dev, layout, M, N, K):
    """Mid-size M (the tile-shape cost model's narrow and 128-wide CTA tiles), N not a
    multiple of the CTA tile and ragged K: sampled rows against the oracle, rows bitwise
    equal to the row computed alone, nothing written outside Y."""
    gi = inputs.gemm_inputs(M, N, K, seed=M + N)
    w = (gi.w_nk if layout == "nk" else gi.w_kn).to(dev)
    buf = torch.full((M + 2, N + 8), 7.0, dtype=torch.bfloat16, device=dev)
    out = buf[1:M + 1, :N]
    bi.matmul(gi.x.to(dev), w, layout, out=out)
    y = out.cpu()
    rows = sorted({0, 63, 64, M // 2, M - 1})
    ref = oracle.matmul(inputs.bf16_bits(gi.x[rows]), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_bf16(y[rows], ref, f"mid-M {M}x{N}x{K} {layout}")
    for i in (0, M - 1):
        alone = bi.matmul(gi.x[i:i + 1].to(dev), w, layout).cpu()
        assert bits_equal(alone, y[i:i + 1]), f"row {i} differs alone"
    assert torch.all(buf[0] == 7.0) and torch.all(buf[M + 1] == 7.0)
    assert torch.all(buf[1:M + 1, N:] == 7.0)


def test_matmul_permutation_and_repeat(dev):
    M, N, K = 300, 512, 1024
    gi = inputs.gemm_inputs(M, N, K, seed=41)
    x, w = gi.x.to(dev), gi.w_nk.to(dev)
    base = bi.matmul(x, w, "nk")
    perm = torch.randperm(M, generator=inputs.generator(42)).to(dev)
    permuted = bi.matmul(x[perm].contiguous(), w, "nk")
    assert bits_equal(permuted, base[perm])
    outs = {bytes(bi.matmul(x, w, "nk").view(torch.int16).cpu().numpy()) for _ in range(100)}
    assert len(outs) == 1


def test_matmul_layouts_agree_bitwise(dev):
    """Both W orientations run the same instruction sequence per element."""
    gi = inputs.gemm_inputs(64, 256, 512, seed=51)
    a = bi.matmul(gi.x.to(dev), gi.w_nk.to(dev), "nk", out_dtype=torch.float32)
    b = bi.matmul(gi.x.to(dev), gi.w_kn.to(dev), "kn", out_dtype=torch.float32)
    assert bits_equal(a, b)


def test_matmul_edges_and_guard_bands(dev):
    gi = inputs.gemm_inputs(3, 40, 96, seed=61)
    x, w = gi.x.to(dev), gi.w_nk.to(dev)
    # strided output inside a sentinel-filled buffer: nothing outside [3, 40] is touched
    buf = torch.full((5, 64), -7.0, dtype=torch.float32, device=dev)
    view = buf[1:4, 8:48]
    bi.matmul(x, w, "nk", out=view)
    ref = oracle.matmul(inputs.bf16_bits(gi.x), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    check_f32(view, ref, _abs_scale(gi.x, gi.w_nk), "strided out")
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask[1:4, 8:48] = False
    assert torch.all(buf[mask] == -7.0)
    # K = 0 writes zeros; M = 0 and N = 0 are no-ops
    z = torch.full((3, 40), 5.0, device=dev)
    bi.matmul(x[:, :0], w[:, :0], "nk", out=z)
    assert torch.all(z == 0)
    bi.matmul(x[:0], w, "nk")
    # unaligned leading dimension: refused before any launch
    xs = torch.zeros(3, 101, dtype=torch.bfloat16, device=dev)[:, :96]
    with pytest.raises(bi.BIError) as e:
        bi.matmul(xs, w, "nk")
    assert e.value.status == bi.BI_ERR_UNSUPPORTED
    assert bi.device_status() == bi.BI_OK


def test_limit_gate_selects_the_configuration(dev):
    """Inside the limit (M <= limit) the invariant single K loop runs, and a row's bits
    equal the row alone; with the limit at 0 this shape (one M-tile, eight 32-column
    tiles) takes a split-K cluster instead ("Fix/speculative shape invariance", Changes:
    dimensions above the limit keep the optimized paths).  Both meet the oracle bar."""
    gi = inputs.gemm_inputs(8, 256, 256, seed=71)
    x, w = gi.x.to(dev), gi.w_nk.to(dev)
    ref = oracle.matmul(inputs.bf16_bits(gi.x), inputs.bf16_bits(gi.w_nk), oracle.W_NK)
    old = bi.get_batch_invariant_limit()
    try:
        bi.set_batch_invariant_limit(0)
        assert bi.matmul_splits(8, 256, 256) > 1
        a = bi.matmul(x, w, "nk", out_dtype=torch.float32)
        bi.set_batch_invariant_limit(8)
        assert bi.matmul_splits(8, 256, 256) == 1
        b = bi.matmul(x, w, "nk", out_dtype=torch.float32)
        alone = bi.matmul(x[3:4].contiguous(), w, "nk", out_dtype=torch.float32)
    finally:
        bi.set_batch_invariant_limit(old)
    check_f32(a, ref, _abs_scale(gi.x, gi.w_nk), "limit 0 (split K)")
    check_f32(b, ref, _abs_scale(gi.x, gi.w_nk), "inside the limit")
    assert bits_equal(alone, b[3:4])
