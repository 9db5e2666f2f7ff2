"""Pins for the oracle's quantized-weight decoding ("Fix/speculative shape invariance",
the tester's comment: affine, mxfp4, mxfp8, nvfp4; "Fix fp quantized matmul corruption
when the quantized dim is not a multiple of 32", Problem: nvfp4 with K = 16 mod 32).

Element and scale codes are pinned against hand-decoded tables from the format
definitions (and FP8 E4M3 against torch's own float8_e4m3fn conversion for all 256
codes); the dequantizer is pinned on the nibble order, group indexing, the affine form
and the K = 1040 tail, so a swapped nibble, an off-by-one group or a dropped bias fails."""
import math

import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs


def test_fp4_e2m1_table():
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    got = oracle.decode_fp4(np.arange(16, dtype=np.uint8))
    assert list(got[:8]) == want and list(got[8:]) == [-v for v in want]
    assert math.copysign(1.0, got[8]) == -1.0  # code 8 is -0


def test_fp8_e4m3_hand_decoded_and_all_codes():
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x7E: 448.0, 0xB8: -1.0, 0xC0: -2.0}
    got = oracle.decode_fp8(np.array(list(cases), dtype=np.uint8))
    assert list(got) == list(cases.values())
    assert np.isnan(oracle.decode_fp8(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    mine = oracle.decode_fp8(codes.numpy())
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(mine), ~ok)
    assert np.array_equal(mine[ok], ref[ok])


def test_e8m0_scales():
    got = oracle.decode_e8m0(np.array([0, 1, 126, 127, 128, 254], dtype=np.uint8))
    assert list(got) == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]
    assert np.isnan(oracle.decode_e8m0(np.array([255], dtype=np.uint8)))[0]


def _bits_of(vals):
    f = np.asarray(vals, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def test_dequantize_nibble_order_and_groups_mxfp4():
    # one row, K = 64: byte b holds elements 2b (low nibble) and 2b+1 (high nibble)
    wq = np.zeros((1, 32), dtype=np.uint8)
    wq[0, 0] = 0x21          # k=0: code 1 (0.5), k=1: code 2 (1.0)
    wq[0, 16] = 0xF7         # k=32: code 7 (6.0), k=33: code 15 (-6.0)
    sc = np.array([[127 + 1, 127 - 2]], dtype=np.uint8)  # group 0: x2, group 1: x1/4
    d = oracle.dequantize(wq, sc, None, oracle.Q_MXFP4, 32, 1, 64)
    vals = (d.astype(np.uint32) << 16).view(np.float32)[0]
    assert vals[0] == 1.0 and vals[1] == 2.0 and vals[2] == 0.0
    assert vals[32] == 1.5 and vals[33] == -1.5 and vals[31] == 0.0


def test_dequantize_nvfp4_tail_and_mxfp8():
    K = 1040  # 65 groups of 16: K = 16 mod 32
    wq, sc, _ = inputs.quant_weights(oracle.Q_NVFP4, 3, K, 16, seed=5)
    d = oracle.dequantize(wq.numpy(), sc.numpy(), None, oracle.Q_NVFP4, 16, 3, K)
    v = (d.astype(np.uint32) << 16).view(np.float32)
    codes = wq.numpy()
    for n, k in ((0, 0), (1, 1039), (2, 1024), (2, 1025)):
        nib = (codes[n, k // 2] >> (4 * (k & 1))) & 15
        want = oracle.decode_fp4(np.array([nib], dtype=np.uint8))[0] * \
            oracle.decode_fp8(sc.numpy()[n, k // 16:k // 16 + 1])[0]
        assert v[n, k] == want
    wq8, sc8, _ = inputs.quant_weights(oracle.Q_MXFP8, 2, 64, 32, seed=6)
    d8 = oracle.dequantize(wq8.numpy(), sc8.numpy(), None, oracle.Q_MXFP8, 32, 2, 64)
    v8 = (d8.astype(np.uint32) << 16).view(np.float32)
    want8 = oracle.decode_fp8(wq8.numpy()[:, :64]) * np.repeat(oracle.decode_e8m0(sc8.numpy()), 32, axis=1)
    assert np.array_equal(v8, want8)


@pytest.mark.parametrize("gs", [32, 64, 128])
def test_dequantize_affine(gs):
    K = 256
    wq, sc, bi_ = inputs.quant_weights(oracle.Q_AFFINE4, 2, K, gs, seed=gs)
    d = oracle.dequantize(wq.numpy(), inputs.bf16_bits(sc), inputs.bf16_bits(bi_),
                          oracle.Q_AFFINE4, gs, 2, K)
    v = (d.astype(np.uint32) << 16).view(np.float32)
    s = sc.float().numpy()
    b = bi_.float().numpy()
    codes = wq.numpy()
    for n, k in ((0, 0), (0, gs), (1, K - 1), (1, gs - 1)):
        q = (codes[n, k // 2] >> (4 * (k & 1))) & 15
        exact = np.float64(s[n, k // gs]) * q + np.float64(b[n, k // gs])
        # fma rounds once to fp32, then to bf16: within one bf16 step of the exact value
        assert abs(v[n, k] - exact) <= abs(exact) * 2.0 ** -8 + 1e-30
    # q = 0 gives the bias itself (exact)
    wq0 = np.zeros_like(wq.numpy())
    d0 = oracle.dequantize(wq0, inputs.bf16_bits(sc), inputs.bf16_bits(bi_), oracle.Q_AFFINE4, gs, 2, K)
    assert np.array_equal(d0[:, ::gs], inputs.bf16_bits(bi_))
    # 8-bit codes: one byte per element
    wq8, sc8, b8 = inputs.quant_weights(oracle.Q_AFFINE8, 1, K, gs, seed=gs + 1)
    d8 = oracle.dequantize(wq8.numpy(), inputs.bf16_bits(sc8), inputs.bf16_bits(b8),
                           oracle.Q_AFFINE8, gs, 1, K)
    v8 = ((d8.astype(np.uint32) << 16).view(np.float32))[0]
    for k in (0, 5, K - 1):
        q = int(wq8.numpy()[0, k])
        exact = np.float64(sc8.float().numpy()[0, k // gs]) * q + np.float64(b8.float().numpy()[0, k // gs])
        assert abs(v8[k] - exact) <= abs(exact) * 2.0 ** -8 + 1e-30


def test_qmatmul_is_matmul_of_dequantized():
    M, N, K = 3, 5, 64
    x = inputs.normal_bf16((M, K), seed=9)
    wq, sc, _ = inputs.quant_weights(oracle.Q_MXFP4, N, K, 32, seed=10)
    y = oracle.qmatmul(inputs.bf16_bits(x), wq.numpy(), sc.numpy(), None, oracle.Q_MXFP4, 32, N)
    d = oracle.dequantize(wq.numpy(), sc.numpy(), None, oracle.Q_MXFP4, 32, N, K)
    xv = inputs.bf16_bits(x).astype(np.uint32) << 16
    dv = d.astype(np.uint32) << 16
    ref = xv.view(np.float32).astype(np.float64) @ dv.view(np.float32).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-5, atol=1e-6)
