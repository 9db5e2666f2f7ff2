"""Pins of the CPU oracle to values the pages print (tests/golden/, each cited there).

The book chapter "Batch-invariant kernels: why temperature-0 decoding is still
nondeterministic" runs CPU listings and prints their output; the oracle's reduction
primitives, RMSNorm and argmax must reproduce those numbers bit for bit.
"""
import random

import numpy as np
import pytest

import oracle
from golden_util import load


def _fmt8(v) -> str:
    return f"{float(v):.8e}"


def test_case1_left_fold_unique_sums():
    """Case 1: 255 distinct left-fold sums of eight cancelling values over 10000 orders."""
    g = load("case1_shuffle_sum.txt")
    vals0 = [1e-10, 1e-5, 1e-2, 1.0]
    vals0 = vals0 + [-v for v in vals0]
    random.seed(42)
    left, builtin = set(), set()
    for _ in range(10_000):
        vals = vals0[:]
        random.shuffle(vals)
        left.add(oracle.left_fold_f64(vals))
        builtin.add(sum(vals))
    assert len(left) == int(g["left_fold_unique"])
    assert repr(min(left)) == g["left_fold_min"]
    assert repr(max(left)) == g["left_fold_max"]
    # the printed control: the compensated builtin sum collapses every order to one value
    assert len(builtin) == int(g["builtin_sum_unique"])


def _case2_vector():
    rng = np.random.default_rng(0)
    return (rng.standard_normal(4096) * 1e3).astype(np.float32)


def test_case2_sequential_and_pairwise():
    g = load("case2_reduction_orders.txt")
    a = _case2_vector()
    assert _fmt8(oracle.sum_sequential_f32(a)) == g["sequential"]
    assert _fmt8(oracle.sum_pairwise_f32(a)) == g["pairwise"]


@pytest.mark.parametrize("splits", [1, 2, 4, 8, 16, 32, 64, 128])
def test_case2_split_k(splits):
    g = load("case2_reduction_orders.txt")
    a = _case2_vector()
    seq = oracle.sum_sequential_f32(a)
    v = oracle.sum_split_f32(a, splits)
    want_sum, want_diff = g[f"split_{splits}"].split()
    assert _fmt8(v) == want_sum
    assert _fmt8(abs(float(v) - float(seq))) == want_diff


def test_case2_split_handles_uneven_chunks():
    """array_split semantics: 10 elements in 3 chunks are 4,3,3 long."""
    a = np.array([1e8, 1, 1, 1, -1e8, 1, 1, 1, 1, 1], dtype=np.float32)
    # chunks [1e8,1,1,1] -> 1e8 ; [-1e8,1,1] -> -1e8 ; [1,1,1] -> 3 ; total 3
    assert float(oracle.sum_split_f32(a, 3)) == 3.0
    # one chunk of everything, sequential: 1e8+1+1+1 = 1e8, -1e8 -> 0, +5 -> 5
    assert float(oracle.sum_split_f32(a, 1)) == 5.0


def _case4_row():
    return np.array([2.0 ** -(i // 64) for i in range(4096)], dtype=np.float32)


def test_case4_sum_of_squares_forward_reverse():
    g = load("case4_rmsnorm.txt")
    row = _case4_row()
    fwd = oracle.sum_squares_f32(row)
    rev = oracle.sum_squares_f32(row[::-1].copy())
    assert _fmt8(fwd) == g["sum_sq_forward"]
    assert _fmt8(rev) == g["sum_sq_reverse"]
    assert _fmt8(abs(float(fwd) - float(rev))) == g["sum_sq_absdiff"]


def test_case4_rmsnorm_heuristic_vs_fixed():
    """The oracle's RMSNorm on the row and on the reversed row reproduces the chapter's
    forward-tree vs reverse-tree comparison exactly (weight 1, eps 1e-6)."""
    g = load("case4_rmsnorm.txt")
    row = _case4_row()
    xb = oracle.bf16_round(row)                       # exact: powers of two
    assert np.array_equal(oracle.bf16_widen(xb), row)
    gamma = oracle.bf16_round(np.ones(4096, dtype=np.float32))
    fwd = oracle.rmsnorm(xb[None, :], gamma, 1e-6)[0]
    rev = oracle.rmsnorm(xb[::-1].copy()[None, :], gamma, 1e-6)[0][::-1]
    assert f"{float(np.max(np.abs(fwd - rev))):.6e}" == g["heuristic_maxdiff"]
    assert int(np.sum(fwd != rev)) == int(g["heuristic_differing"])
    # fixed tree: the same row alone and inside a batch of 16 gives the same bits
    batch = np.stack([xb] + [oracle.bf16_round(np.float32(1 + i) * row) for i in range(15)])
    in_batch = oracle.rmsnorm(batch, gamma, 1e-6)[0]
    assert f"{float(np.max(np.abs(fwd - in_batch))):.6e}" == g["fixed_maxdiff"]
    assert np.array_equal(fwd.view(np.uint32), in_batch.view(np.uint32))


def _tiled_matvec(a_row, B, tile_k):
    """The chapter's Case 3/5 accumulation (numpy BLAS for each tile, fp32 adds)."""
    acc = np.zeros(B.shape[1], dtype=np.float32)
    for t in range(0, a_row.shape[0], tile_k):
        acc = acc + (a_row[t:t + tile_k] @ B[t:t + tile_k]).astype(np.float32)
    return acc


def test_case3_batch_aware_tile_changes_row0():
    """Harness pin: a batch-size-dependent K tile changes row 0; a fixed tile does not.
    (The partial products go through numpy's BLAS, as in the chapter.)"""
    g = load("case3_batch_matmul.txt")
    D = 4096
    A0 = np.linspace(-1000, 1000, 2048 * D, dtype=np.float32)[:D]
    B = np.linspace(-1000, 1000, D * D, dtype=np.float32).reshape(D, D)
    full = _tiled_matvec(A0, B, int(g["tile_full"]))
    one = _tiled_matvec(A0, B, int(g["tile_one"]))
    assert f"{float(np.max(np.abs(full - one))):.4f}" == g["diff_heuristic"]
    fixed_a = _tiled_matvec(A0, B, 256)
    fixed_b = _tiled_matvec(A0.copy(), B, 256)
    assert f"{float(np.max(np.abs(fixed_a - fixed_b))):.4f}" == g["diff_fixed"]


def test_case5_greedy_token_under_load_uses_oracle_argmax():
    """The oracle's argmax reproduces the chapter's greedy tokens under three K-tile
    choices, and a single token under the fixed tile."""
    g = load("case5_load_nondet.txt")
    D, V = 4096, 8192
    token = np.linspace(-50, 50, D, dtype=np.float32)
    W = np.linspace(-1, 1, D * V, dtype=np.float32).reshape(D, V)
    ref = _tiled_matvec(token, W, 256)
    toks_h = []
    for row in g["row"]:
        load_, tile, tok, dmax, top1 = row.split()
        logits = _tiled_matvec(token, W, int(tile))
        t = oracle.argmax_f32(logits)
        toks_h.append(t)
        assert t == int(tok)
        assert f"{float(np.max(np.abs(logits - ref))):.4f}" == dmax
        assert f"{float(logits[t]):.4f}" == top1
    assert sorted(set(toks_h)) == [int(x) for x in g["heuristic_tokens"].split()]
    fixed = {oracle.argmax_f32(_tiled_matvec(token, W, 256)) for _ in range(2)}
    assert sorted(fixed) == [int(x) for x in g["fixed_tokens"].split()]
