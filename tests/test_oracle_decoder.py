"""Pins for the oracle's decoder glue (positions, rotary embedding, SwiGLU, residual add,
argmax NaN rule) and for its composition into the greedy-trace decoder stack.  Each pin
checks the oracle against something other than itself: closed-form values, identities
of the mathematics, numpy's complex arithmetic, or numpy fp64 on special cases where a
branch of the stack reduces to a closed form."""
import numpy as np
import pytest
import torch

import oracle
from oracle.decoder import OracleDecoder
from invariant_bi_matmul_gb300 import inputs
from golden_util import load

GOLD = load("decoder_glue_closed_forms.txt")


def _floats(key):
    return np.array([float(v) for v in GOLD[key].split()])


def _bits(vals):
    return inputs.bf16_bits(torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16))


def _widen(bits):
    return oracle.bf16_widen(bits).astype(np.float64)


# ------------------------------------------------------------------------ positions

def test_positions_follow_the_causal_block_rule():
    # sequence 0 holds 5 tokens, its block is the last 2 (positions 3, 4); sequence 1
    # holds 3 tokens, its block is the last 1 (position 2)
    assert oracle.positions(np.array([5, 3]), np.array([0, 2, 3])).tolist() == [3, 4, 2]
    assert oracle.positions(np.array([5, 3])).tolist() == [4, 2]      # decode
    assert oracle.positions(np.array([4]), np.array([0, 4])).tolist() == [0, 1, 2, 3]


# --------------------------------------------------------------------------- rotary

def test_rope_hand_example():
    x = _bits(_floats("rope_d4_x")).reshape(1, 1, 4)
    y = oracle.rope(x, np.array([int(GOLD["rope_d4_pos"])], dtype=np.int32),
                    float(GOLD["rope_d4_theta"]))
    np.testing.assert_allclose(y.ravel(), _floats("rope_d4_y"), rtol=1e-14, atol=1e-14)


def test_rope_position_zero_is_identity():
    x = inputs.bf16_bits(inputs.normal_bf16((3, 4, 64), seed=11))
    y = oracle.rope(x, np.zeros(3, dtype=np.int32), 500000.0)
    assert np.array_equal(y, _widen(x))


def test_rope_d2_is_complex_rotation():
    # D = 2: one pair at frequency 1, i.e. multiplication of x0 + i x1 by e^{i pos}
    x = inputs.bf16_bits(inputs.normal_bf16((50, 1, 2), seed=12))
    pos = np.arange(0, 5000, 100, dtype=np.int32)
    y = oracle.rope(x, pos, 500000.0)
    xw = _widen(x)
    z = (xw[:, 0, 0] + 1j * xw[:, 0, 1]) * np.exp(1j * pos.astype(np.float64))
    np.testing.assert_allclose(y[:, 0, 0], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 1], z.imag, rtol=0, atol=1e-12)


def test_rope_matches_complex_form_and_keeps_pair_norms():
    T, H, D = 6, 3, 128
    x = inputs.bf16_bits(inputs.normal_bf16((T, H, D), seed=13))
    pos = np.array([0, 1, 7, 100, 4097, 8447], dtype=np.int32)
    y = oracle.rope(x, pos, 500000.0)
    xw = _widen(x)
    z = xw[..., :D // 2] + 1j * xw[..., D // 2:]
    freq = np.power(500000.0, -np.arange(D // 2) * 2.0 / D)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    np.testing.assert_allclose(y[..., :D // 2], zr.real, atol=1e-9)
    np.testing.assert_allclose(y[..., D // 2:], zr.imag, atol=1e-9)
    n_in = xw[..., :D // 2] ** 2 + xw[..., D // 2:] ** 2
    n_out = y[..., :D // 2] ** 2 + y[..., D // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12, atol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    D = 64
    q = inputs.bf16_bits(inputs.normal_bf16((1, 1, D), seed=14))
    k = inputs.bf16_bits(inputs.normal_bf16((1, 1, D), seed=15))
    ref = None
    for m, n in [(10, 3), (7, 0), (1007, 1000), (8199, 8192)]:
        qm = oracle.rope(q, np.array([m], dtype=np.int32), 10000.0).ravel()
        kn = oracle.rope(k, np.array([n], dtype=np.int32), 10000.0).ravel()
        s = float(qm @ kn)
        ref = s if ref is None else ref
        assert abs(s - ref) < 1e-9 * max(1.0, abs(ref))


# --------------------------------------------------------------------------- SwiGLU

def test_swiglu_closed_forms():
    y = oracle.swiglu(_bits(_floats("swiglu_g")), _bits(_floats("swiglu_u")))
    np.testing.assert_allclose(y, _floats("swiglu_y"), rtol=1e-15, atol=0)


def test_silu_reflection_identity():
    # silu(x) - silu(-x) = x for every x (u = 1)
    g = inputs.bf16_bits(inputs.normal_bf16((4096,), std=4.0, seed=16))
    neg = g ^ np.uint16(0x8000)
    one = _bits(np.ones(4096))
    d = oracle.swiglu(g, one) - oracle.swiglu(neg, one)
    np.testing.assert_allclose(d, _widen(g), rtol=1e-13, atol=1e-13)


def test_swiglu_limits():
    y = oracle.swiglu(_bits([100.0, -100.0, 30.0]), _bits([3.0, 1.0, -2.0]))
    assert y[0] == 300.0 and abs(y[1]) < 1e-40 and abs(y[2] + 60.0) < 1e-10


# ------------------------------------------------------------------------------ add

def test_add_is_the_exact_sum():
    a = inputs.bf16_bits(inputs.normal_bf16((1000,), std=10.0, seed=17))
    b = inputs.bf16_bits(inputs.normal_bf16((1000,), std=0.01, seed=18))
    assert np.array_equal(oracle.add(a, b), _widen(a) + _widen(b))
    assert oracle.add(_bits([1.5]), _bits([2.25]))[0] == 3.75


# --------------------------------------------------------------------- argmax / NaN

@pytest.mark.parametrize("vals,want", [([np.nan, 1.0, 2.0], 2), ([np.nan, np.nan], 0),
                                       ([1.0, np.nan, 1.0], 0), ([-np.inf, np.nan], 0),
                                       ([np.nan, -np.inf, -np.inf], 1), ([3.0, 5.0, 5.0], 1)])
def test_argmax_ranks_nan_lowest_and_breaks_ties_low(vals, want):
    assert oracle.argmax_f32(np.array(vals, dtype=np.float32)) == want


# ------------------------------------------------------------- decoder composition

CFG = inputs.DecoderConfig(hidden=64, heads=4, kv_heads=2, head_dim=16, inter=96, layers=1,
                           vocab=50, context=0, eps=1e-5, theta=10000.0)


def _weights(seed, zero=()):
    w = {k: inputs.bf16_bits(v) for k, v in
         inputs.decoder_weights(CFG, seed, std=0.1, norm_std=0.1).items()}
    for k in zero:
        w[k] = np.zeros_like(w[k])
    return w


def _f(bits):
    return _widen(bits)


def _np_rmsnorm(h, gamma, eps):
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * gamma


def _decoder(w, pages=4):
    return OracleDecoder(CFG, w, num_pages=pages, block_table=np.arange(pages).reshape(1, pages))


def _close(got, want, tol=2e-2):
    err = np.abs(got - want)
    assert np.all(err <= tol + 1e-2 * np.abs(want)), float(err.max())


def test_zeroed_branches_leave_the_embedding_on_the_residual_stream():
    w = _weights(21, zero=("l0.wo", "l0.w_down"))
    logits = _decoder(w).forward([7], seq_lens=[1], cu_q=[0, 1])
    x = _np_rmsnorm(_f(w["embed"][7]), _f(w["final_norm"]), CFG.eps)
    _close(logits[0], _f(w["lm_head"]) @ x)


def test_one_key_attention_returns_v_through_the_o_projection():
    # a lone token attends only to itself: the attention output is its own V (per KV head,
    # shared by the query heads of its group), whatever q, k and the rotation are
    w = _weights(22, zero=("l0.w_down",))
    logits = _decoder(w).forward([3], seq_lens=[1], cu_q=[0, 1])
    e = _f(w["embed"][3])
    x = _np_rmsnorm(e, _f(w["l0.attn_norm"]), CFG.eps)
    v = (_f(w["l0.wv"]) @ x).reshape(CFG.kv_heads, CFG.head_dim)
    group = CFG.heads // CFG.kv_heads
    a = np.concatenate([v[h // group] for h in range(CFG.heads)])
    h1 = e + _f(w["l0.wo"]) @ a
    _close(logits[0], _f(w["lm_head"]) @ _np_rmsnorm(h1, _f(w["final_norm"]), CFG.eps))


def test_mlp_branch_is_down_of_silu_gate_times_up():
    w = _weights(23, zero=("l0.wo",))
    logits = _decoder(w).forward([11], seq_lens=[1], cu_q=[0, 1])
    e = _f(w["embed"][11])
    x = _np_rmsnorm(e, _f(w["l0.mlp_norm"]), CFG.eps)
    g, u = _f(w["l0.w_gate"]) @ x, _f(w["l0.w_up"]) @ x
    h1 = e + _f(w["l0.w_down"]) @ (g / (1 + np.exp(-g)) * u)
    _close(logits[0], _f(w["lm_head"]) @ _np_rmsnorm(h1, _f(w["final_norm"]), CFG.eps))


def test_block_of_four_equals_four_single_steps_bitwise():
    # the oracle evaluates every row on its own, so a token inside a causal block and
    # the same token alone give the same bits
    w = _weights(24)
    toks = [5, 9, 1, 30]
    one = _decoder(w)
    singles = np.stack([one.forward([t], seq_lens=[i + 1], cu_q=[0, 1])[0]
                        for i, t in enumerate(toks)])
    block = _decoder(w).forward(toks, seq_lens=[4], cu_q=[0, 4])
    assert np.array_equal(singles.view(np.uint32), block.view(np.uint32))
