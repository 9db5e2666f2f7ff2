"""Pins for the oracle's row-wise log-softmax and mean (book chapter "Batch-invariant
kernels...", Sources: the mean and log-softmax overrides; textbook definitions).

Each pin is a closed form or an invariant of the definition, chosen so that a plausible
slip fails one of them: a dropped max shift overflows the large-magnitude rows; a sum
over the wrong count breaks the uniform row; a sign or operand swap breaks the two-point
closed form; a missing -inf rule breaks the masked rows."""
import math

import numpy as np

import oracle


def test_log_softmax_uniform_row_is_minus_log_n():
    for n in (1, 2, 7, 4096):
        for c in (0.0, -3.5, 1e6):
            y = oracle.log_softmax(np.full(n, c, dtype=np.float32))
            assert np.allclose(y, -math.log(n), rtol=0, atol=1e-12)


def test_log_softmax_two_point_closed_form():
    # [0, ln 3]: softmax = [1/4, 3/4]
    y = oracle.log_softmax(np.array([0.0, math.log(3.0)], dtype=np.float32))
    x1 = float(np.float32(math.log(3.0)))
    assert abs(y[0] - (-math.log(1.0 + math.exp(x1)))) < 1e-15
    assert abs(y[1] - (x1 - math.log(1.0 + math.exp(x1)))) < 1e-15
    assert abs(y[0] + math.log(4.0)) < 1e-7 and abs(y[1] - math.log(0.75)) < 1e-7


def test_log_softmax_normalises_and_is_shift_invariant():
    rng = np.random.default_rng(5)
    # multiples of 2^-8 below 64 in magnitude: x + 64 is exact in fp32
    x = (np.round(np.clip(rng.normal(0, 4, (6, 333)), -60, 60) * 256) / 256).astype(np.float32)
    y = oracle.log_softmax(x)
    assert np.allclose(np.exp(y).sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(y <= 0)
    # adding a constant exactly representable at these magnitudes changes nothing
    y2 = oracle.log_softmax(x + np.float32(64.0))
    assert np.allclose(y, y2, rtol=0, atol=1e-9)
    # differences of outputs are differences of inputs
    assert np.allclose(y[:, 1:] - y[:, :1], x[:, 1:].astype(np.float64) - x[:, :1], atol=1e-12)


def test_log_softmax_large_magnitudes_do_not_overflow():
    y = oracle.log_softmax(np.array([1000.0, 0.0], dtype=np.float32))
    assert abs(y[0] - (-math.log1p(math.exp(-1000.0)))) < 1e-15
    assert abs(y[1] - (-1000.0)) < 1e-12
    y = oracle.log_softmax(np.array([-3e38, -3e38], dtype=np.float32))
    assert np.allclose(y, -math.log(2.0))


def test_log_softmax_special_values():
    ninf = -np.inf
    y = oracle.log_softmax(np.array([0.0, ninf, 0.0], dtype=np.float32))
    assert y[1] == -np.inf and np.allclose(y[[0, 2]], -math.log(2.0))
    assert np.all(np.isnan(oracle.log_softmax(np.array([1.0, np.nan, 2.0], dtype=np.float32))))
    assert np.all(np.isnan(oracle.log_softmax(np.array([ninf, ninf], dtype=np.float32))))
    assert np.all(np.isnan(oracle.log_softmax(np.array([np.inf, 0.0], dtype=np.float32))))


def test_mean_closed_forms():
    for n in (1, 2, 5, 1000, 4097):
        assert oracle.mean(np.arange(n, dtype=np.float32))[0] == (n - 1) / 2
        assert oracle.mean(np.full(n, 3.25, dtype=np.float32))[0] == 3.25
    # bf16 bits: 1.0 = 0x3F80, 2.0 = 0x4000, -0.5 = 0xBF00
    bits = np.array([[0x3F80, 0x4000, 0xBF00, 0x4000]], dtype=np.uint16)
    assert oracle.mean(bits, bf16=True)[0] == (1.0 + 2.0 - 0.5 + 2.0) / 4
    # rows are independent
    x = np.stack([np.arange(8, dtype=np.float32), -np.arange(8, dtype=np.float32)])
    assert list(oracle.mean(x)) == [3.5, -3.5]
