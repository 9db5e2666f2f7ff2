"""Pins of the CPU oracle to mathematics: closed forms, exact-integer cases, special
cases that reduce to a library routine (numpy fp64), brute force on tiny inputs.

Each test is built so that a plausible mistake (dropped term, wrong sign or index,
transposed operand, eps outside the root, off-by-one causal mask, wrong GQA head,
wrong page lookup) fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs

U = 2.0 ** -24  # fp32 unit roundoff


def bits(t):
    return inputs.bf16_bits(t)


def f64(t):
    return t.to(torch.float64).numpy()


# ------------------------------------------------------------------------ bf16 round

def test_bf16_round_matches_library_cast_and_specials():
    g = inputs.generator(11)
    vals = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 10)
    specials = torch.tensor([0.0, -0.0, 1.0, -1.0, float("inf"), float("-inf"), 3.4e38, -3.4e38,
                             1e-40, -1e-40, 1.00390625, 1.01171875, 1.0078125 + 2 ** -20,
                             2.0 ** -133, 65504.0, 3.0e38 * 1.13])
    x = torch.cat([vals, specials]).to(torch.float32)
    # ties: halfway between two bf16 values, both parities of the kept bit
    ties = torch.tensor([0x3F808000, 0x3F818000, 0xBF808000, 0x7F7F8000], dtype=torch.int64)
    ties = ties.to(torch.int32).view(torch.float32)
    x = torch.cat([x, ties])
    mine = oracle.bf16_round(x.numpy())
    lib = bits(x.to(torch.bfloat16))
    assert np.array_equal(mine, lib)
    nan = oracle.bf16_round(np.array([np.nan, -np.nan], dtype=np.float32))
    assert np.all(np.isnan(oracle.bf16_widen(nan)))


def test_argmax_lowest_index_on_ties_and_library():
    v = np.array([1.0, 3.0, 2.0, 3.0, -np.inf], dtype=np.float32)
    assert oracle.argmax_f32(v) == 1
    rng = np.random.default_rng(5)
    for _ in range(20):
        w = rng.integers(-3, 4, size=257).astype(np.float32)
        assert oracle.argmax_f32(w) == int(np.argmax(w))   # numpy: first occurrence


# --------------------------------------------------------------------------- matmul

@pytest.mark.parametrize("layout", [oracle.W_NK, oracle.W_KN])
def test_matmul_vs_fp64_within_gamma_k(layout):
    M, N, K = 5, 7, 300
    gi = inputs.gemm_inputs(M, N, K, seed=3)
    w = gi.w_nk if layout == oracle.W_NK else gi.w_kn
    y = oracle.matmul(bits(gi.x), bits(w), layout).astype(np.float64)
    X, Wt = f64(gi.x), f64(gi.w_nk).T               # Wt is [K, N]
    ref = X @ Wt
    scale = np.abs(X) @ np.abs(Wt)
    assert np.all(np.abs(y - ref) <= (K + 2) * U * scale)


def test_matmul_layouts_give_identical_bits():
    gi = inputs.gemm_inputs(4, 33, 129, seed=4)
    a = oracle.matmul(bits(gi.x), bits(gi.w_nk), oracle.W_NK)
    b = oracle.matmul(bits(gi.x), bits(gi.w_kn), oracle.W_KN)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_matmul_dropped_or_transposed_term_detected():
    """Negative control on the checker above: a K-1 sum or a transposed W is caught."""
    M, N, K = 3, 5, 64
    gi = inputs.gemm_inputs(M, N, K, seed=9)
    X, Wt = f64(gi.x), f64(gi.w_nk).T
    scale = np.abs(X) @ np.abs(Wt)
    dropped = X[:, :-1] @ Wt[:-1, :]
    assert np.any(np.abs(dropped - X @ Wt) > (K + 2) * U * scale)
    y = oracle.matmul(bits(gi.x), bits(gi.w_nk), oracle.W_NK).astype(np.float64)
    assert np.max(np.abs(y - X @ Wt)) < 1e-4


def test_matmul_exact_integers_bit_exact():
    """Small integers times powers of two: every partial sum is exact in fp32, so any
    summation order (the oracle's, numpy's, a tensor core's) gives the same value."""
    M, N, K = 6, 40, 512
    x = inputs.small_int_bf16((M, K), -8, 8, 0, seed=1)
    w = inputs.small_int_bf16((N, K), -8, 8, -3, seed=2)
    y = oracle.matmul(bits(x), bits(w), oracle.W_NK)
    ref = f64(x) @ f64(w).T
    assert np.array_equal(y.astype(np.float64), ref)


def test_matmul_strides_and_empty_k():
    M, N, K, ldx, ldw, ldy = 3, 4, 10, 16, 24, 7
    rng = np.random.default_rng(0)
    xs = oracle.bf16_round(rng.standard_normal(M * ldx).astype(np.float32))
    ws = oracle.bf16_round(rng.standard_normal(N * ldw).astype(np.float32))
    y = oracle.matmul_strided(xs, ldx, ws, ldw, oracle.W_NK, M, N, K, ldy).reshape(M, ldy)
    X = oracle.bf16_widen(xs).reshape(M, ldx)[:, :K].astype(np.float64)
    W = oracle.bf16_widen(ws).reshape(N, ldw)[:, :K].astype(np.float64)
    assert np.allclose(y[:, :N], X @ W.T, rtol=1e-5, atol=1e-5)
    assert np.all(np.isnan(y[:, N:]))                # padding of y never written
    y0 = oracle.matmul_strided(xs, ldx, ws, ldw, oracle.W_NK, M, N, 0, ldy).reshape(M, ldy)
    assert np.all(y0[:, :N] == 0.0)


# -------------------------------------------------------------------------- rmsnorm

def test_rmsnorm_constant_row_closed_form():
    H, c, eps = 1024, 1.5, 1e-5
    x = torch.full((1, H), c, dtype=torch.bfloat16)
    gamma = inputs.normal_bf16((H,), 1.0, 0.1, seed=5)
    y = oracle.rmsnorm(bits(x), bits(gamma), eps)[0].astype(np.float64)
    ref = c / np.sqrt(c * c + eps) * f64(gamma)
    assert np.allclose(y, ref, rtol=4 * 2 ** -23, atol=0)


def test_rmsnorm_eps_zero_powers_of_two_exact():
    """x = +-2^3, eps = 0: mean(x^2) = 64 exactly, inv = 1/8 exactly, y = +-gamma."""
    H = 4096
    g = inputs.generator(6)
    signs = torch.where(torch.rand(H, generator=g) < 0.5, -1.0, 1.0)
    x = (signs * 8.0).to(torch.bfloat16)[None]
    gamma = inputs.normal_bf16((H,), 1.0, 0.1, seed=7)
    y = oracle.rmsnorm(bits(x), bits(gamma), 0.0)[0]
    assert np.array_equal(y.astype(np.float64), signs.numpy() * f64(gamma))


def test_rmsnorm_vs_fp64_with_large_eps():
    """eps = 0.5 is large enough that eps outside the root, or a wrong gamma index, or a
    sum over the wrong axis, is far outside the tolerance."""
    B, H, eps = 4, 777, 0.5
    x, gamma = inputs.rmsnorm_inputs(B, H, seed=8, std=1.0)
    y = oracle.rmsnorm(bits(x), bits(gamma), eps).astype(np.float64)
    X, G = f64(x), f64(gamma)
    ref = X / np.sqrt(np.mean(X * X, axis=1, keepdims=True) + eps) * G
    assert np.allclose(y, ref, rtol=1e-5, atol=1e-6)
    wrong = X / (np.sqrt(np.mean(X * X, axis=1, keepdims=True)) + eps) * G
    assert not np.allclose(wrong, ref, rtol=1e-3, atol=1e-4)


def test_rmsnorm_row_independent_of_batch():
    x, gamma = inputs.rmsnorm_inputs(16, 512, seed=9)
    full = oracle.rmsnorm(bits(x), bits(gamma), 1e-5)
    for i in (0, 7, 15):
        one = oracle.rmsnorm(bits(x[i:i + 1]), bits(gamma), 1e-5)[0]
        assert np.array_equal(one.view(np.uint32), full[i].view(np.uint32))


# --------------------------------------------------------------- paged KV / attention

def _gather(cache, bt_row, L):
    """[pages,Hkv,page,D] -> [Hkv, L, D] for one sequence (numpy, independent)."""
    page = cache.shape[2]
    idx = np.arange(L)
    pages = bt_row[idx // page]
    return np.transpose(cache[pages, :, idx % page, :], (1, 0, 2))


def _reference_attention(p: inputs.PagedInputs, Hq, scale):
    """Brute-force fp64 causal softmax attention from numpy primitives."""
    kc = f64(p.k_cache)
    vc = f64(p.v_cache)
    q = f64(p.q)
    Hkv = kc.shape[1]
    G = Hq // Hkv
    T, _, D = q.shape
    out = np.zeros((T, Hq, D))
    lse = np.zeros((T, Hq))
    bt = p.block_table.numpy()
    for b in range(p.B):
        L = int(p.seq_lens[b])
        c0, c1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        K = _gather(kc, bt[b], L)
        V = _gather(vc, bt[b], L)
        for j in range(c1 - c0):
            pos = L - (c1 - c0) + j
            for h in range(Hq):
                s = K[h // G, :pos + 1] @ q[c0 + j, h] * scale
                m = s.max()
                e = np.exp(s - m)
                out[c0 + j, h] = e @ V[h // G, :pos + 1] / e.sum()
                lse[c0 + j, h] = m + np.log(e.sum())
    return out, lse


def _appended(p):
    return oracle.kv_append(bits(p.k_new), bits(p.v_new), bits(p.k_cache), bits(p.v_cache),
                            p.block_table.numpy(), p.seq_lens.numpy(), p.cu_q.numpy(), p.page_size)


def _with_cache(p, kc, vc):
    import dataclasses
    return dataclasses.replace(p, k_cache=torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16),
                               v_cache=torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16))


def test_kv_append_scatters_to_the_right_slots():
    p = inputs.paged_inputs([5, 70, 130], [1, 3, 4], Hq=4, Hkv=2, D=16, seed=10, page_size=8)
    kc, vc = _appended(p)
    k0, v0 = bits(p.k_cache), bits(p.v_cache)
    changed = np.zeros(kc.shape[:3], dtype=bool)
    bt = p.block_table.numpy()
    for b in range(p.B):
        L, c0, c1 = int(p.seq_lens[b]), int(p.cu_q[b]), int(p.cu_q[b + 1])
        for j in range(c1 - c0):
            pos = L - (c1 - c0) + j
            pg, sl = bt[b, pos // 8], pos % 8
            assert np.array_equal(kc[pg, :, sl], bits(p.k_new)[c0 + j])
            assert np.array_equal(vc[pg, :, sl], bits(p.v_new)[c0 + j])
            changed[pg, :, sl] = True
    assert np.array_equal(kc[~changed], k0[~changed])
    assert np.array_equal(vc[~changed], v0[~changed])


def test_attention_vs_fp64_brute_force_causal_gqa_paged():
    Hq, Hkv, D = 8, 2, 32
    p = inputs.paged_inputs([5, 70, 130, 1], [1, 3, 4, 1], Hq=Hq, Hkv=Hkv, D=D, seed=11,
                            page_size=8)
    kc, vc = _appended(p)
    p = _with_cache(p, kc, vc)
    scale = 1.0 / np.sqrt(D)
    out, lse = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                                p.cu_q.numpy(), Hq, scale)
    ref, ref_lse = _reference_attention(p, Hq, scale)
    assert np.allclose(out, ref, rtol=2e-5, atol=2e-5)
    assert np.allclose(lse, ref_lse, rtol=1e-5, atol=1e-5)


def test_attention_zero_keys_give_mean_of_visible_values_exactly():
    """K = 0: every score is 0, p = 1, l = n; with integer V and n a power of two the
    result sum(v)/n is exact, so the oracle must match it bit for bit."""
    Hq = Hkv = 2
    D = 8
    p = inputs.paged_inputs([16], [4], Hq=Hq, Hkv=Hkv, D=D, seed=12, page_size=4)
    kc = np.zeros_like(bits(p.k_cache))
    vi = inputs.small_int_bf16(p.v_cache.shape, -20, 20, 0, seed=13)
    vc = bits(vi)
    out, lse = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                                p.cu_q.numpy(), Hq, 0.125)
    V = _gather(f64(vi), p.block_table.numpy()[0], 16)
    # query j=3 sees 16 keys (a power of two); j=1 sees 14 (not exact, allclose)
    for h in range(Hq):
        assert np.array_equal(out[3, h].astype(np.float64), V[h, :16].mean(axis=0))
        assert np.allclose(out[1, h], V[h, :14].mean(axis=0), rtol=1e-6, atol=1e-6)
        assert lse[3, h] == np.float32(np.log(np.float32(16)))


def test_attention_single_key_returns_v0():
    p = inputs.paged_inputs([1], [1], Hq=4, Hkv=4, D=64, seed=14)
    kc, vc = _appended(p)
    out, _ = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                              p.cu_q.numpy(), 4, 0.125)
    assert np.array_equal(out[0].astype(np.float64), f64(p.v_new)[0])


def test_attention_dominant_key_selects_its_value():
    Hq = Hkv = 1
    D = 16
    p = inputs.paged_inputs([40], [1], Hq=Hq, Hkv=Hkv, D=D, seed=15, page_size=8, kv_std=0.01)
    kc, vc = _appended(p)
    t = 23
    pg, sl = int(p.block_table[0, t // 8]), t % 8
    qv = f64(p.q)[0, 0]
    kc[pg, 0, sl] = bits(torch.tensor(qv * 400.0 / np.dot(qv, qv), dtype=torch.float32)
                         .to(torch.bfloat16))
    out, _ = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                              p.cu_q.numpy(), Hq, 1.0)
    assert np.allclose(out[0, 0], oracle.bf16_widen(vc[pg, 0, sl]), atol=1e-6)


def test_attention_causal_mask_boundary():
    """Query j of a block sees keys 0..pos exactly: changing key pos+1 leaves it alone,
    changing key pos moves it."""
    Hq = Hkv = 1
    D = 16
    p = inputs.paged_inputs([20], [4], Hq=Hq, Hkv=Hkv, D=D, seed=16, page_size=8)
    kc, vc = _appended(p)
    args = (p.block_table.numpy(), p.seq_lens.numpy(), p.cu_q.numpy(), Hq, 0.25)
    base, _ = oracle.attention(bits(p.q), kc, vc, *args)
    pos0 = 20 - 4  # query 0 sits at position 16
    for t, same in ((pos0 + 1, True), (pos0, False)):
        vc2 = vc.copy()
        pg, sl = int(p.block_table[0, t // 8]), t % 8
        vc2[pg, 0, sl] = oracle.bf16_round(np.full(D, 100.0, dtype=np.float32))
        out, _ = oracle.attention(bits(p.q), kc, vc2, *args)
        assert np.array_equal(out[0], base[0]) == same


def test_attention_page_permutation_is_transparent():
    Hq, Hkv, D = 4, 2, 16
    p = inputs.paged_inputs([37, 9], [2, 1], Hq=Hq, Hkv=Hkv, D=D, seed=17, page_size=8)
    kc, vc = _appended(p)
    args = (p.seq_lens.numpy(), p.cu_q.numpy(), Hq, 0.3)
    out_a, lse_a = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), *args)
    # rebuild the same logical sequences with pages in identity order
    bt = p.block_table.numpy()
    order = [int(x) for x in bt.ravel() if x >= 0]
    kc2 = kc.copy()
    vc2 = vc.copy()
    bt2 = np.full_like(bt, -1)
    for new, old in enumerate(order):
        kc2[new] = kc[old]
        vc2[new] = vc[old]
    it = iter(range(len(order)))
    for b in range(bt.shape[0]):
        for i in range(bt.shape[1]):
            if bt[b, i] >= 0:
                bt2[b, i] = next(it)
    out_b, lse_b = oracle.attention(bits(p.q), kc2, vc2, bt2, *args)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_attention_gqa_head_grouping():
    """V of KV head i is the constant i: query head h must read KV head h // (Hq/Hkv)."""
    Hq, Hkv, D = 8, 2, 16
    p = inputs.paged_inputs([24], [2], Hq=Hq, Hkv=Hkv, D=D, seed=18, page_size=8)
    kc, _ = _appended(p)
    vc = np.empty_like(kc)
    for i in range(Hkv):
        vc[:, i] = oracle.bf16_round(np.full(vc[:, i].shape, float(i), dtype=np.float32))
    out, _ = oracle.attention(bits(p.q), kc, vc, p.block_table.numpy(), p.seq_lens.numpy(),
                              p.cu_q.numpy(), Hq, 0.25)
    for h in range(Hq):
        assert np.all(out[:, h] == float(h // (Hq // Hkv)))


def test_attention_row_matches_full():
    Hq, Hkv, D = 4, 2, 32
    p = inputs.paged_inputs([50, 17], [3, 2], Hq=Hq, Hkv=Hkv, D=D, seed=19, page_size=16)
    kc, vc = _appended(p)
    bt, sl, cq = p.block_table.numpy(), p.seq_lens.numpy(), p.cu_q.numpy()
    out, lse = oracle.attention(bits(p.q), kc, vc, bt, sl, cq, Hq, 0.2)
    o, l = oracle.attention_row(bits(p.q), kc, vc, bt, sl, cq, 1, 1, 3, Hq, 0.2)
    t = int(cq[1]) + 1
    assert np.array_equal(o, out[t, 3]) and np.float32(l) == lse[t, 3]
