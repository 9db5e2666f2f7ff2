"""The order-sensitive GEMM operands (inputs.adversarial_operand) on the CPU: they are exact
in their format, their cancelling pairs cancel, and -- the point of them -- two
reasonable ways of summing the same products give different fp32 results for most
output elements, so a GPU test comparing fp32 bits across M would see any change in how
an instruction groups its 16-wide K slices.  Summation orders from the book chapter
"Batch-invariant kernels...", Case 2 (sequential, pairwise and split sums of one vector
differ in fp32)."""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_operands_are_exact_and_pairs_cancel(dtype):
    K = 256
    x = inputs.adversarial_operand(8, K, seed=1, role="x", dtype=dtype)
    w = inputs.adversarial_operand(8, K, seed=2, role="w", dtype=dtype)
    assert torch.equal(x.double().to(dtype), x) and torch.isfinite(x.double()).all()
    xd, wd = x.double(), w.double()
    for a in (0, 8):
        s = xd[:, None, a::16] * wd[None, :, a::16] + xd[:, None, a + 1::16] * wd[None, :, a + 1::16]
        assert torch.all(s == 0)
        assert torch.all(xd[:, a::16].abs() >= (2.0 ** 7))
    tiny = 2.0 ** (-126 if dtype == torch.bfloat16 else -14)
    assert torch.all(xd[:, 5::16].abs() < tiny) and torch.all(xd[:, 5::16] != 0)
    assert torch.all(wd[:, 6::16].abs() < tiny) and torch.all(wd[:, 6::16] != 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_summation_order_is_visible_in_fp32(dtype):
    """Sequential fp32 (the oracle's order) against a fold of exact 16-term slice sums
    (what an instruction with a wider internal adder would do): most elements differ."""
    K, R = 4096, 16
    x = inputs.adversarial_operand(R, K, seed=3, role="x", dtype=dtype).double().numpy()
    w = inputs.adversarial_operand(R, K, seed=4, role="w", dtype=dtype).double().numpy()
    differ = 0
    for i in range(R):
        for j in range(R):
            prods = (x[i] * w[j]).astype(np.float32)
            seq = oracle.sum_sequential_f32(prods)
            slices = (x[i] * w[j]).reshape(-1, 16).sum(axis=1)   # exact in fp64 here
            acc = np.float32(0)
            for s in slices.astype(np.float32):
                acc = np.float32(acc + s)
            differ += int(np.float32(seq) != acc)
    assert differ > R * R // 2, differ
