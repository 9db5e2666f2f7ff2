"""Greedy-trace decoder: a Llama-style decoder stack run through libbi, either token by
token or in greedy speculative-verification blocks, to show that the greedy token trace
does not depend on the batch a sequence is decoded in or on the verify width.

Pages: "Fix/speculative shape invariance" (ml-explore/mlx PR 4279), section Problem
(evaluating a token alone and inside a short verification block must give identical
results, else greedy decoding diverges); book chapter "Batch-invariant kernels: why
temperature-0 decoding is still nondeterministic", Case 5 (the same request's greedy
token under different server loads).

Every arithmetic step runs in libbi kernels (embedding, RMSNorm, the projections, RoPE,
KV append, verify attention, residual adds, SwiGLU, LM head, argmax).  This module only
allocates device tensors with torch, keeps the per-sequence bookkeeping (how many tokens
each cache holds, the next input token) and applies the greedy acceptance rule of
speculative decoding on the host: a drafted token is kept while it equals the greedy
token the verify block computed at its position; the first mismatch is replaced by that
greedy token, which ends the step.

Contexts: each sequence starts with ``cfg.context`` tokens already in its KV caches.
``prefill`` computes them from a prompt through the same kernels, in causal blocks of
``prefill_width`` tokens (blocks wider than a verify block go through the chunked-prefill
attention, which reduces every query exactly as the verify kernel does, so the cache
bits do not depend on the block width); ``start`` instead loads synthetic cache rows
(seeded N(0,1) keys and values per sequence and layer, written with bi_kv_append), for
small checks against the oracle.  Either way a sequence's context depends only on the
sequence, never on the batch it runs in.

The traces are batch invariant only while every call is inside the batch-invariant
limit: matmuls of up to ``max_batch * max_width`` rows and verify blocks of up to
``max_width`` tokens.  An ``invariant=True`` decoder (the default) refuses to run a block
the current limit does not cover; ``invariant=False`` runs whatever the limit selects.
"""
from __future__ import annotations

import math
from typing import Callable, List, Optional, Sequence

import torch

from . import (ATTN_MAX_Q, add, argmax, attn_workspace_size, embedding, kv_append, matmul,
               prefill_attn, rmsnorm, rope, swiglu, verify_block, within_batch_invariant_limit)
from .inputs import PAGE_SIZE, DecoderConfig, decoder_context, decoder_first_token, page_permutation

Drafter = Callable[[int, List[int], int], List[int]]


class GreedyDecoder:
    """A decoder stack with paged KV caches for up to ``max_batch`` sequences of up to
    ``max_len`` tokens, evaluated in blocks of up to ``max_width`` tokens per sequence
    (``prefill_width`` for prompts, default ``max_width``)."""

    def __init__(self, cfg: DecoderConfig, weights: dict, max_batch: int, max_len: int,
                 max_width: int = 4, device="cuda", page_seed: int = 0,
                 invariant: bool = True, prefill_width: int = 0):
        self.cfg, self.w = cfg, weights
        self.invariant = invariant
        self.dev = torch.device(device)
        self.max_batch, self.max_len, self.max_width = max_batch, max_len, max_width
        self.prefill_width = max(prefill_width, max_width)
        c = cfg
        pps = math.ceil(max_len / PAGE_SIZE)
        self.num_pages = max_batch * pps
        # physical pages in a seeded random order, so sequences' pages interleave
        self.block_table = page_permutation(self.num_pages, page_seed).view(
            max_batch, pps).contiguous().to(self.dev)
        shape = (self.num_pages, c.kv_heads, PAGE_SIZE, c.head_dim)
        self.k_cache = [torch.zeros(shape, dtype=torch.bfloat16, device=self.dev)
                        for _ in range(c.layers)]
        self.v_cache = [torch.zeros(shape, dtype=torch.bfloat16, device=self.dev)
                        for _ in range(c.layers)]
        T = max_batch * self.prefill_width     # activations: the widest block
        Td = max_batch * max_width               # logits: decoding blocks only
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        self.h = torch.empty(T, c.hidden, **bf)
        self.x = torch.empty(T, c.hidden, **bf)
        self.o = torch.empty(T, c.hidden, **bf)
        self.q = torch.empty(T, c.heads * c.head_dim, **bf)
        self.k = torch.empty(T, c.kv_heads * c.head_dim, **bf)
        self.v = torch.empty(T, c.kv_heads * c.head_dim, **bf)
        self.attn = torch.empty(T, c.heads, c.head_dim, **bf)
        self.g = torch.empty(T, c.inter, **bf)
        self.u = torch.empty(T, c.inter, **bf)
        self.a = torch.empty(T, c.inter, **bf)
        self.logits = torch.empty(Td, c.vocab, dtype=torch.float32, device=self.dev)
        self.tokens = torch.empty(Td, dtype=torch.int32, device=self.dev)
        self.ids = torch.empty(T, dtype=torch.int32, device=self.dev)
        self.seq_lens = torch.empty(max_batch, dtype=torch.int32, device=self.dev)
        self.cu_q = torch.empty(max_batch + 1, dtype=torch.int32, device=self.dev)
        self.ws = torch.empty(attn_workspace_size(T, c.heads, c.head_dim, max_len),
                              dtype=torch.uint8, device=self.dev)
        self.scale = 1.0 / math.sqrt(c.head_dim)
        self.batch = 0
        self.cached: List[int] = []
        self.last: List[int] = []

    # ----------------------------------------------------------------- sequences
    def start(self, seq_ids: Sequence[int], seed: int,
              context_fn: Optional[Callable[[int, int], tuple]] = None,
              first_tokens: Optional[Sequence[int]] = None) -> None:
        """Loads the sequences' contexts into cache slots 0..len(seq_ids)-1.
        context_fn(seq_id, layer) -> (k, v) bf16 [context, Hkv, D]; by default seeded
        N(0,1) rows drawn on the device."""
        c = self.cfg
        B = len(seq_ids)
        if not 1 <= B <= self.max_batch:
            raise ValueError(f"batch must be in [1, {self.max_batch}]")
        if c.context + self.max_width > self.max_len:
            raise ValueError("max_len leaves no room after the context")
        if context_fn is None:
            def context_fn(sid, layer):
                return decoder_context(c, sid, layer, seed, device=self.dev)
        one = torch.tensor([c.context], dtype=torch.int32, device=self.dev)
        cu = torch.tensor([0, c.context], dtype=torch.int32, device=self.dev)
        for b, sid in enumerate(seq_ids):
            if c.context == 0:
                break
            for layer in range(c.layers):
                k, v = context_fn(sid, layer)
                kv_append(k.to(self.dev).contiguous(), v.to(self.dev).contiguous(),
                          self.k_cache[layer], self.v_cache[layer],
                          self.block_table[b:b + 1], one, cu)
        self.batch = B
        self.cached = [c.context] * B
        self.last = (list(first_tokens) if first_tokens is not None else
                     [decoder_first_token(c, sid, seed) for sid in seq_ids])

    # ------------------------------------------------------------------- forward
    def forward(self, ids: Sequence[int], q_lens: Sequence[int],
                logits: bool = True) -> Optional[torch.Tensor]:
        """Runs one ragged block: sequence b contributes q_lens[b] tokens (its next input
        token first) at positions cached[b] .. cached[b]+q_lens[b]-1; their K/V are
        appended to the caches.  Returns the greedy tokens (device int32 [T]); the fp32
        logits stay in ``self.logits[:T]``.  With logits=False (prefill) the final norm,
        LM head and argmax are skipped and None is returned."""
        c, w = self.cfg, self.w
        B = self.batch
        T = len(ids)
        widest = self.max_width if logits else self.prefill_width
        if len(q_lens) != B or sum(q_lens) != T or max(q_lens) > widest:
            raise ValueError("one block of 1..max_width (prefill: prefill_width) tokens per "
                             "sequence")
        lens = [self.cached[b] + q_lens[b] for b in range(B)]
        if max(lens) > self.max_len:
            raise ValueError("sequence longer than max_len")
        if self.invariant and not (within_batch_invariant_limit(T) and
                                   within_batch_invariant_limit(max(q_lens))):
            raise RuntimeError(f"the batch-invariant limit does not cover a block of {T} tokens "
                               f"(widest {max(q_lens)}): raise it with "
                               "set_batch_invariant_limit, or build the decoder with "
                               "invariant=False")
        cu = [0]
        for q in q_lens:
            cu.append(cu[-1] + q)
        self.seq_lens[:B].copy_(torch.tensor(lens, dtype=torch.int32), non_blocking=False)
        self.cu_q[:B + 1].copy_(torch.tensor(cu, dtype=torch.int32), non_blocking=False)
        self.ids[:T].copy_(torch.tensor(list(ids), dtype=torch.int32), non_blocking=False)
        sl, cq, bt = self.seq_lens[:B], self.cu_q[:B + 1], self.block_table[:B]
        h, x, o = self.h[:T], self.x[:T], self.o[:T]
        q = self.q[:T].view(T, c.heads, c.head_dim)
        k = self.k[:T].view(T, c.kv_heads, c.head_dim)
        v = self.v[:T].view(T, c.kv_heads, c.head_dim)
        attn, g, u, a = self.attn[:T], self.g[:T], self.u[:T], self.a[:T]
        embedding(w["embed"], self.ids[:T], out=h)
        for i in range(c.layers):
            p = f"l{i}."
            rmsnorm(h, w[p + "attn_norm"], c.eps, out=x)
            matmul(x, w[p + "wq"], out=self.q[:T])
            matmul(x, w[p + "wk"], out=self.k[:T])
            matmul(x, w[p + "wv"], out=self.v[:T])
            rope(q, sl, cq, c.theta)
            rope(k, sl, cq, c.theta)
            kv_append(k, v, self.k_cache[i], self.v_cache[i], bt, sl, cq)
            # blocks wider than a verify block: the chunked-prefill kernel (same bits)
            attend = verify_block if max(q_lens) <= ATTN_MAX_Q else prefill_attn
            attend(q, self.k_cache[i], self.v_cache[i], bt, sl, cq, max_q=max(q_lens),
                   max_seq_len=max(lens), scale=self.scale, out=attn, want_lse=False,
                   workspace=self.ws)
            matmul(attn.view(T, c.heads * c.head_dim), w[p + "wo"], out=o)
            add(h, o, out=h)
            rmsnorm(h, w[p + "mlp_norm"], c.eps, out=x)
            matmul(x, w[p + "w_gate"], out=g)
            matmul(x, w[p + "w_up"], out=u)
            swiglu(g, u, out=a)
            matmul(a, w[p + "w_down"], out=o)
            add(h, o, out=h)
        if not logits:
            return None
        rmsnorm(h, w["final_norm"], c.eps, out=x)
        matmul(x, w["lm_head"], out=self.logits[:T])
        return argmax(self.logits[:T], out=self.tokens[:T])

    # ------------------------------------------------------------------ prefill
    def prefill(self, prompts: Sequence[Sequence[int]], width: Optional[int] = None) -> None:
        """Puts prompts (one per cache slot 0..len-1, all of one length P) through the
        stack: tokens 0..P-2 in causal blocks of `width` (default prefill_width), their
        K/V into the caches; token P-1 becomes the first input of decoding."""
        B = len(prompts)
        P = len(prompts[0])
        width = width or self.prefill_width
        if not 1 <= B <= self.max_batch or any(len(p) != P for p in prompts) or P < 1:
            raise ValueError("1..max_batch prompts of one length >= 1")
        if not 1 <= width <= self.prefill_width or P - 1 + self.max_width > self.max_len:
            raise ValueError("width or prompt length out of range")
        self.batch = B
        self.cached = [0] * B
        for s0 in range(0, P - 1, width):
            n = min(width, P - 1 - s0)
            ids = [t for p in prompts for t in p[s0:s0 + n]]
            self.forward(ids, [n] * B, logits=False)
            self.cached = [x + n for x in self.cached]
        self.last = [p[P - 1] for p in prompts]

    def snapshot(self):
        """The caches and per-sequence state, to run several decodings from one context."""
        return ([k.clone() for k in self.k_cache], [v.clone() for v in self.v_cache],
                self.batch, list(self.cached), list(self.last))

    def restore(self, snap, batch: Optional[int] = None) -> None:
        """Back to a snapshot, keeping its first `batch` sequences (cache slots)."""
        ks, vs, B, cached, last = snap
        for dst, src in zip(self.k_cache, ks):
            dst.copy_(src)
        for dst, src in zip(self.v_cache, vs):
            dst.copy_(src)
        self.batch = B if batch is None else batch
        if not 1 <= self.batch <= B:
            raise ValueError("batch must be in [1, snapshot batch]")
        self.cached = cached[:self.batch]
        self.last = last[:self.batch]

    # ------------------------------------------------------------------- drivers
    def decode(self, steps: int) -> List[List[int]]:
        """Token-by-token greedy decoding: `steps` tokens per sequence."""
        B = self.batch
        traces: List[List[int]] = [[] for _ in range(B)]
        for _ in range(steps):
            toks = self.forward(self.last, [1] * B).tolist()
            for b in range(B):
                traces[b].append(toks[b])
                self.cached[b] += 1
                self.last[b] = toks[b]
        return traces

    def speculate(self, steps: int, width: int, drafter: Drafter):
        """Greedy speculative decoding with verify blocks of `width` tokens: the next
        input token plus width-1 drafted ones.  A sequence that already has `steps`
        tokens keeps going with one-token blocks until every sequence has them, so
        blocks of different widths share the batch.  Returns (traces of `steps` tokens
        per sequence, number of forward passes, drafted tokens accepted).  Needs
        max_len >= context + 2*steps + width."""
        if not 1 <= width <= self.max_width:
            raise ValueError(f"width must be in [1, {self.max_width}]")
        B = self.batch
        history = [[self.last[b]] for b in range(B)]
        traces: List[List[int]] = [[] for _ in range(B)]
        blocks = accepted = 0
        while min(len(t) for t in traces) < steps:
            q_lens = [width if len(traces[b]) < steps else 1 for b in range(B)]
            drafts = [list(drafter(b, history[b], q_lens[b] - 1))[:q_lens[b] - 1]
                      if q_lens[b] > 1 else [] for b in range(B)]
            ids = []
            for b in range(B):
                ids.append(self.last[b])
                ids.extend(drafts[b])
            greedy = self.forward(ids, q_lens).tolist()
            blocks += 1
            t0 = 0
            for b in range(B):
                gb = greedy[t0:t0 + q_lens[b]]
                t0 += q_lens[b]
                n = 0
                while n < q_lens[b] - 1 and drafts[b][n] == gb[n]:
                    n += 1
                new = drafts[b][:n] + [gb[n]]
                accepted += n
                traces[b].extend(new)
                history[b].extend(new)
                self.cached[b] += n + 1
                self.last[b] = gb[n]
        return [t[:steps] for t in traces], blocks, accepted


def lookup_drafter(b: int, history: List[int], n: int) -> List[int]:
    """Prompt-lookup drafting: find the latest earlier occurrence of the last token and
    propose the tokens that followed it (padded with the last token)."""
    last = history[-1]
    for i in range(len(history) - 2, -1, -1):
        if history[i] == last:
            follow = history[i + 1:i + 1 + n]
            return follow + [last] * (n - len(follow))
    return [last] * n


def random_drafter(vocab: int, seed: int) -> Drafter:
    """Seeded random drafts (almost always rejected: every block ends at its first
    token)."""
    g = torch.Generator().manual_seed(int(seed))

    def draft(b: int, history: List[int], n: int) -> List[int]:
        return torch.randint(0, vocab, (n,), generator=g).tolist()
    return draft


def reference_drafter(reference: List[List[int]], corrupt_fraction: float, vocab: int,
                      seed: int = 0) -> Drafter:
    """Drafts the continuation a reference run produced, with a seeded pseudo-random
    `corrupt_fraction` of the trace positions replaced by another token, so blocks end
    at varying depths (0 replays the reference: every draft is accepted)."""
    def corrupted(t: int) -> bool:
        hsh = ((t + 1) * 2654435761 + seed * 40503) & 0xffffffff
        return (hsh >> 8) % 1000 < corrupt_fraction * 1000

    def draft(b: int, history: List[int], n: int) -> List[int]:
        done = len(history) - 1  # tokens emitted so far
        ref = reference[b]
        out = []
        for i in range(n):
            t = done + i
            tok = ref[t] if t < len(ref) else history[-1]
            if corrupted(t):
                tok = (tok + 1) % vocab
            out.append(tok)
        return out
    return draft
