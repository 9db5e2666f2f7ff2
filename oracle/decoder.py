"""Plain CPU forward pass of the greedy-trace decoder stack, composed from the oracle's
functions (TEST INFRASTRUCTURE ONLY; the product library never imports it).

The stack is the Llama-3-8B-shaped decoder of the full-decoder workload: per layer
RMSNorm -> q/k/v projections -> rotary embedding -> KV-cache append -> causal paged
attention -> o projection -> residual add -> RMSNorm -> gate/up projections -> SwiGLU ->
down projection -> residual add; then a final RMSNorm and the LM head (fp32 logits),
greedy argmax with the lowest index on ties.  Pages: "Fix/speculative shape
invariance" (ml-explore/mlx PR 4279), section Problem (one token alone vs inside a
verification block must give identical results); book chapter "Batch-invariant
kernels: why temperature-0 decoding is still nondeterministic", Case 5 (the greedy
token under different loads).

Every activation between two operations is stored as bf16 (the model's dtype), each
operation computing from bf16 inputs and rounding its own result once; the logits stay
fp32.  This is the oracle's reading of a bf16 model and the GPU path stores the same
tensors in the same dtypes, so the two differ only by summation order inside each
operation.  Each step below is one oracle call or a numpy gather / reshape.

Weights are a dict of bf16 bit arrays (uint16), named as ``inputs.decoder_weights``
names them: ``embed`` [V,hidden], ``lm_head`` [V,hidden], ``final_norm`` [hidden] and
per layer ``l{i}.attn_norm``, ``l{i}.wq`` [Hq*D,hidden], ``l{i}.wk`` / ``l{i}.wv``
[Hkv*D,hidden], ``l{i}.wo`` [hidden,Hq*D], ``l{i}.mlp_norm``, ``l{i}.w_gate`` /
``l{i}.w_up`` [I,hidden], ``l{i}.w_down`` [hidden,I] (all nn.Linear [out,in]).
"""
from __future__ import annotations

import numpy as np

from . import (W_NK, add, argmax_f32, attention, kv_append, matmul, positions, rmsnorm, rope,
               swiglu, to_bf16)


class OracleDecoder:
    """Holds the weights and one paged KV cache per layer (uint16 [pages,Hkv,page,D])."""

    def __init__(self, cfg, weights: dict, num_pages: int, block_table: np.ndarray,
                 page_size: int = 64):
        self.cfg = cfg
        self.w = weights
        self.page = page_size
        self.block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        shape = (num_pages, cfg.kv_heads, page_size, cfg.head_dim)
        self.k_cache = [np.zeros(shape, dtype=np.uint16) for _ in range(cfg.layers)]
        self.v_cache = [np.zeros(shape, dtype=np.uint16) for _ in range(cfg.layers)]

    def append_context(self, layer: int, slot: int, k: np.ndarray, v: np.ndarray):
        """Writes a sequence's context K/V rows (uint16 [n,Hkv,D], positions 0..n-1) into
        the cache pages of block-table row `slot` of one layer."""
        n = k.shape[0]
        self.k_cache[layer], self.v_cache[layer] = kv_append(
            k, v, self.k_cache[layer], self.v_cache[layer], self.block_table[slot:slot + 1],
            np.array([n], dtype=np.int32), np.array([0, n], dtype=np.int32), self.page)

    def forward(self, tokens, seq_lens, cu_q) -> np.ndarray:
        """Logits fp32 [T,V] for a ragged block: tokens int [T]; sequence b's tokens are
        cu_q[b]..cu_q[b+1]-1 and end at position seq_lens[b]-1 (its cache holds the
        earlier positions).  The block's K/V are appended to the caches."""
        c, w = self.cfg, self.w
        tokens = np.asarray(tokens, dtype=np.int64)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
        T = tokens.size
        pos = positions(seq_lens, cu_q)
        scale = 1.0 / np.sqrt(c.head_dim)
        h = w["embed"][tokens]                                   # bf16 [T,hidden]
        for i in range(c.layers):
            p = f"l{i}."
            x = to_bf16(rmsnorm(h, w[p + "attn_norm"], c.eps))
            q = to_bf16(matmul(x, w[p + "wq"], W_NK)).reshape(T, c.heads, c.head_dim)
            k = to_bf16(matmul(x, w[p + "wk"], W_NK)).reshape(T, c.kv_heads, c.head_dim)
            v = to_bf16(matmul(x, w[p + "wv"], W_NK)).reshape(T, c.kv_heads, c.head_dim)
            q = to_bf16(rope(q, pos, c.theta))
            k = to_bf16(rope(k, pos, c.theta))
            self.k_cache[i], self.v_cache[i] = kv_append(
                k, v, self.k_cache[i], self.v_cache[i], self.block_table, seq_lens, cu_q,
                self.page)
            a, _ = attention(q, self.k_cache[i], self.v_cache[i], self.block_table, seq_lens,
                             cu_q, c.heads, scale)
            a = to_bf16(a).reshape(T, c.heads * c.head_dim)
            o = to_bf16(matmul(a, w[p + "wo"], W_NK))
            h = to_bf16(add(h, o))
            x = to_bf16(rmsnorm(h, w[p + "mlp_norm"], c.eps))
            g = to_bf16(matmul(x, w[p + "w_gate"], W_NK))
            u = to_bf16(matmul(x, w[p + "w_up"], W_NK))
            act = to_bf16(swiglu(g, u))
            d = to_bf16(matmul(act, w[p + "w_down"], W_NK))
            h = to_bf16(add(h, d))
        x = to_bf16(rmsnorm(h, w["final_norm"], c.eps))
        return matmul(x, w["lm_head"], W_NK)

    @staticmethod
    def greedy(logits: np.ndarray) -> np.ndarray:
        """Greedy token of every logits row (lowest index among equal maxima)."""
        return np.array([argmax_f32(row) for row in logits], dtype=np.int64)
