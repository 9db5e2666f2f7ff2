"""Pins for the oracle's IEEE binary16 path (16-bit inputs of matmul and RMSNorm).

binary16 widening is pinned by hand-decoded patterns from the format definition and by
every one of the 65,536 patterns against numpy's own conversion; matmul16 / rmsnorm16
with binary16 inputs are pinned by exact-integer cases, by agreement with the bf16 path
on values both formats represent exactly, and by a closed form."""
import math

import numpy as np

import oracle


def test_f16_hand_decoded_patterns():
    cases = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0400: 2.0 ** -14,
             0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24, 0x3555: 1365 / 4096,
             0x8000: -0.0, 0x7C00: math.inf, 0xFC00: -math.inf}
    got = oracle.f16_widen(np.array(list(cases), dtype=np.uint16))
    for (bits, want), g in zip(cases.items(), got):
        assert g == want and math.copysign(1, g) == math.copysign(1, want), hex(bits)
    assert np.isnan(oracle.f16_widen(np.array([0x7E00, 0xFC01], dtype=np.uint16))).all()


def test_f16_every_pattern_matches_numpy():
    h = np.arange(65536, dtype=np.uint16)
    a = oracle.f16_widen(h)
    b = h.view(np.float16).astype(np.float32)
    ok = ~np.isnan(b)
    assert np.array_equal(np.isnan(a), ~ok)
    assert np.array_equal(a[ok].view(np.uint32), b[ok].view(np.uint32))


def _f16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def _bf16_exact(a):
    """bf16 bits of values that bf16 represents exactly (checked)."""
    f = np.asarray(a, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), f)
    return bits


def test_matmul16_f16_exact_integers_and_bf16_agreement():
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, (5, 40)).astype(np.float64)
    w = rng.integers(-8, 9, (7, 40)).astype(np.float64)
    want = x @ w.T                                    # every partial sum is an exact integer
    y = oracle.matmul16(_f16(x), _f16(w), oracle.W_NK, oracle.F16)
    assert np.array_equal(y, want.astype(np.float32))
    y_kn = oracle.matmul16(_f16(x), _f16(w.T.copy()), oracle.W_KN, oracle.F16)
    assert np.array_equal(y_kn, y)
    # halves and quarters: exact in both formats, so both paths give the same fp32 bits
    xq = rng.integers(-64, 65, (4, 33)) / 4.0
    wq = rng.integers(-64, 65, (6, 33)) / 8.0
    a = oracle.matmul16(_f16(xq), _f16(wq), oracle.W_NK, oracle.F16)
    b = oracle.matmul16(_bf16_exact(xq), _bf16_exact(wq), oracle.W_NK, oracle.BF16)
    assert np.array_equal(a, b)
    assert np.array_equal(b, oracle.matmul(_bf16_exact(xq), _bf16_exact(wq), oracle.W_NK))


def test_rmsnorm16_f16_closed_form_and_bf16_agreement():
    # a constant row c: ss/H = c^2, so y = c / sqrt(c^2 + eps) * gamma; with eps = 0 and
    # c, gamma powers of two every step is exact
    H = 64
    for c, gm in ((2.0, 0.5), (-0.25, 4.0)):
        y = oracle.rmsnorm16(_f16(np.full((1, H), c)), _f16(np.full(H, gm)), 0.0, oracle.F16)
        assert np.all(y == np.float32(math.copysign(gm, c)))
    rng = np.random.default_rng(4)
    x = rng.integers(-32, 33, (3, 48)) / 8.0
    g = rng.integers(1, 9, 48) / 4.0
    a = oracle.rmsnorm16(_f16(x), _f16(g), 1e-6, oracle.F16)
    b = oracle.rmsnorm16(_bf16_exact(x), _bf16_exact(g), 1e-6, oracle.BF16)
    assert np.array_equal(a, b)
    assert np.array_equal(b, oracle.rmsnorm(_bf16_exact(x), _bf16_exact(g), 1e-6))


def test_matmul_f32_exact_and_library_agreement():
    """fp32 inputs: integers give exact results; a random case agrees with numpy's fp64
    product of the same values (the oracle accumulates exact products in fp64)."""
    rng = np.random.default_rng(6)
    x = rng.integers(-1000, 1001, (4, 50)).astype(np.float32)
    w = rng.integers(-1000, 1001, (6, 50)).astype(np.float32)
    want = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.array_equal(oracle.matmul_f32(x, w, oracle.W_NK), want)
    assert np.array_equal(oracle.matmul_f32(x, w.T.copy(), oracle.W_KN), want)
    xr = rng.normal(size=(3, 700)).astype(np.float32)
    wr = rng.normal(size=(5, 700)).astype(np.float32)
    ref = xr.astype(np.float64) @ wr.astype(np.float64).T
    assert np.allclose(oracle.matmul_f32(xr, wr, oracle.W_NK), ref, rtol=0, atol=1e-10)


def test_rmsnorm_f32_matches_16bit_path_on_shared_values():
    rng = np.random.default_rng(7)
    x = rng.integers(-32, 33, (3, 48)) / 8.0
    g = rng.integers(1, 9, 48) / 4.0
    a = oracle.rmsnorm_f32(x.astype(np.float32), g.astype(np.float32), 1e-6)
    b = oracle.rmsnorm16(_bf16_exact(x), _bf16_exact(g), 1e-6, oracle.BF16)
    assert np.array_equal(a, b)
