"""Rows of bi_matmul compared across M on fp32 output bits, with operands built so that
any change in how an instruction groups or rounds the products of a 16-wide K slice
would change the result (inputs.adversarial_operand: exactly cancelling pairs of large
products beside small terms, subnormal inputs, products in fp32's subnormal range).

The kernel's instruction height (64 rows for tiles of at most 64 rows, else 128) and
width (32 .. 256 columns) and its CTA tile follow M.  The invariance the pages ask for
(book chapter "Batch-invariant kernels...", Case 6, matmul row, which names a smaller
instruction at small M as a way to break it; "Fix/speculative shape invariance", Problem)
then rests on each output element's sum not depending on the instruction's shape.  These
tests pin that on the fp32 accumulator itself -- bf16 rounding would hide most
one-ulp accumulator differences -- for every height, every width the schedule picks at
K = 4096 and 14,336 (the down projection of the pages' decoder stack), both W layouts,
bf16 and binary16 operands, and one quantized format.
"""
import numpy as np
import pytest
import torch

from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")

# M = 1 .. 64: one 64-row instruction; 65 .. 128: one 128-row instruction; 129: two
# M-tiles; 512, 1024, 2048: 64-, 128- and 256-column tiles (256 x 256 CTA tiles at 2048)
M_SWEEP = (1, 2, 8, 63, 64, 65, 127, 128, 129, 256, 512, 1024, 2048)
ALONE = (63, 64, 127, 128, 1000, 1999)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("K", [4096, 14336])
def test_adversarial_rows_fp32_bits_across_M(dev, dtype, layout, K):
    N = 4096
    x = inputs.adversarial_operand(2048, K, seed=K + 1, role="x", dtype=dtype).to(dev)
    w_nk = inputs.adversarial_operand(N, K, seed=K + 2, role="w", dtype=dtype)
    w = (w_nk if layout == "nk" else w_nk.t().contiguous()).to(dev)
    full32 = bi.matmul(x, w, layout, out_dtype=torch.float32)
    full16 = bi.matmul(x, w, layout)
    assert torch.isfinite(full32).all()
    for M in M_SWEEP:
        xm = x[:M].contiguous()
        assert bits_equal(bi.matmul(xm, w, layout, out_dtype=torch.float32), full32[:M]), \
            f"fp32 rows differ at M={M}"
        assert bits_equal(bi.matmul(xm, w, layout), full16[:M]), f"rows differ at M={M}"
    for i in ALONE:
        alone = bi.matmul(x[i:i + 1].contiguous(), w, layout, out_dtype=torch.float32)
        assert bits_equal(alone, full32[i:i + 1]), f"row {i} differs alone"
    # and each row equals itself under a batch permutation (rows land in other lanes)
    perm = torch.randperm(300, generator=inputs.generator(K)).to(dev)
    y = bi.matmul(x[perm].contiguous(), w, layout, out_dtype=torch.float32)
    assert bits_equal(y, full32[:300][perm])
    assert bi.device_status() == bi.BI_OK


def test_adversarial_rows_quantized_fp32_bits_across_M(dev):
    """mxfp4 codes under E8M0 scales spanning 2^-20 .. 2^20, order-sensitive X."""
    N, K, gs = 4096, 4096, 32
    x = inputs.adversarial_operand(2048, K, seed=91, role="x").to(dev)
    wq, _, _ = inputs.quant_weights(inputs.Q_MXFP4, N, K, gs, seed=92)
    g = inputs.generator(93)
    sc = torch.randint(127 - 20, 127 + 21, (N, K // gs), generator=g, dtype=torch.int32)
    sc = sc.to(torch.uint8).to(dev)
    args = (wq.to(dev), sc, "mxfp4", gs, K)
    full = bi.qmatmul(x, *args, out_dtype=torch.float32)
    for M in M_SWEEP:
        part = bi.qmatmul(x[:M].contiguous(), *args, out_dtype=torch.float32)
        assert bits_equal(part, full[:M]), f"quantized fp32 rows differ at M={M}"
    for i in ALONE:
        alone = bi.qmatmul(x[i:i + 1].contiguous(), *args, out_dtype=torch.float32)
        assert bits_equal(alone, full[i:i + 1]), f"quantized row {i} differs alone"
    assert bi.device_status() == bi.BI_OK
