"""Seeded synthetic inputs shaped like the workloads the pages describe.

This module holds none of the method's arithmetic: it only draws random numbers
(``torch.Generator`` seeded per call), casts them to bf16 and lays them out.  Both the
CUDA path and the CPU oracle are fed from here, so neither depends on the other.

Workload shapes (the pages' configurations):
  * tiny check: x ``[M,256]`` N(0,1), M in {1,2,4,8}; W ``[256,256]`` N(0,0.02);
    gamma N(1,0.1), eps 1e-6; attention with 4 heads, head_dim 64, 128 cached tokens.
  * GEMM: K=N=4096, X N(0,1), W N(0,0.02), M in {1,2,4,8,16,64,256,2048}.
  * RMSNorm: hidden 8192, x N(0, std 3) with 1% of elements (independent Bernoulli
    draws) multiplied by 50 before the bf16 cast, gamma N(1,0.1), eps 1e-5.
  * attention: 32 query heads, 8 KV heads, head_dim 128, K/V/Q N(0,1), paged cache with
    64-token pages whose physical order is a random permutation.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

PAGE_SIZE = 64


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, mean: float = 0.0, std: float = 1.0, seed: int = 0) -> torch.Tensor:
    """N(mean, std) drawn in fp32 on the CPU, cast to bf16 (round to nearest even)."""
    t = torch.randn(*shape, generator=generator(seed), dtype=torch.float32)
    return (t * std + mean).to(torch.bfloat16)


def small_int_bf16(shape, lo: int, hi: int, exp2: int = 0, seed: int = 0) -> torch.Tensor:
    """Integers in [lo, hi] times 2**exp2, exactly representable in bf16 (|v| <= 256)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=generator(seed), dtype=torch.int32)
    return (t.to(torch.float32) * (2.0 ** exp2)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (for the C oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


# ------------------------------------------------- order-sensitive GEMM operands

# Per dtype: mantissa bits, exponent range of the ordinary values, exponent of the large
# cancelling values, and the subnormal step of the format.
_ADV = {torch.bfloat16: (7, -10, 10, 10, -133), torch.float16: (10, -8, 7, 7, -24)}


def adversarial_operand(rows: int, K: int, seed: int, role: str,
                        dtype=torch.bfloat16) -> torch.Tensor:
    """A [rows, K] operand whose dot products expose how a multiply-accumulate unit groups
    and rounds the terms of a 16-wide K slice.  In every slice of 16:
      * positions 0,1 and 8,9 hold a cancelling pair: X repeats one large value at k and
        k+1 (role "x"), W holds a large value and its negation (role "w"), so the two
        products (about 2^20 for bf16, 2^14 for f16) cancel exactly for every row and
        column, and whatever small terms were added next to them survive or not by the
        order and width of the additions;
      * position 5 (role "x") or 6 (role "w") holds a subnormal value of the format (one
        step of 2^-133 for bf16, 2^-24 for f16, times 1..127), which meets an ordinary
        value of the other operand;
      * position 12 holds, for bf16, a value near 2^-64 (X) or 2^-70 (W), so that product
        falls in fp32's subnormal range;
      * the rest are +-(1 + m/2^p) * 2^e with e uniform in a wide range (bf16 -10..10,
        f16 -8..7), so products span about 2^-20 .. 2^20.
    Values are drawn as integers and assembled exactly; nothing is rounded."""
    if role not in ("x", "w"):
        raise ValueError("role is 'x' or 'w'")
    pbits, emin, emax, big, sub = _ADV[dtype]
    g = generator(seed)
    sign = torch.randint(0, 2, (rows, K), generator=g).to(torch.float64) * 2 - 1
    mant = 1 + torch.randint(0, 1 << pbits, (rows, K), generator=g).to(torch.float64) / (1 << pbits)
    expo = torch.randint(emin, emax + 1, (rows, K), generator=g).to(torch.float64)
    v = sign * mant * torch.pow(2.0, expo)
    k = torch.arange(K) % 16
    for a in (0, 8):
        first, second = (k == a), (k == a + 1)
        big_vals = sign[:, first] * mant[:, first] * 2.0 ** big
        v[:, first] = big_vals
        v[:, second[:K]] = big_vals[:, :int(second.sum())] * (1.0 if role == "x" else -1.0)
    steps = torch.randint(1, 128, (rows, K), generator=g).to(torch.float64)
    ks = 5 if role == "x" else 6
    v[:, k == ks] = (sign * steps * 2.0 ** sub)[:, k == ks]
    if dtype == torch.bfloat16:
        tiny = -64 if role == "x" else -70
        v[:, k == 12] = (sign * mant * 2.0 ** tiny)[:, k == 12]
    return v.to(dtype)


# ----------------------------------------------------------------------------- GEMM

@dataclass
class GemmInputs:
    x: torch.Tensor      # [M, K] bf16
    w_nk: torch.Tensor   # [N, K] bf16 (nn.Linear weight, "transposed B")
    w_kn: torch.Tensor   # [K, N] bf16, the same matrix stored naturally


def gemm_inputs(M: int, N: int, K: int, seed: int, x_std: float = 1.0,
                w_std: float = 0.02) -> GemmInputs:
    x = normal_bf16((M, K), 0.0, x_std, seed=seed * 1000003 + 1)
    w_nk = normal_bf16((N, K), 0.0, w_std, seed=seed * 1000003 + 2)
    return GemmInputs(x=x, w_nk=w_nk, w_kn=w_nk.t().contiguous())


# -------------------------------------------------------------------------- RMSNorm

def rmsnorm_inputs(B: int, H: int, seed: int, std: float = 3.0, outlier_p: float = 0.01,
                   outlier_scale: float = 50.0):
    """x [B,H] bf16 with independent outliers, gamma [H] bf16 N(1, 0.1)."""
    g = generator(seed)
    x = torch.randn(B, H, generator=g, dtype=torch.float32) * std
    if outlier_p > 0:
        mask = torch.rand(B, H, generator=g) < outlier_p
        x = torch.where(mask, x * outlier_scale, x)
    gamma = torch.randn(H, generator=g, dtype=torch.float32) * 0.1 + 1.0
    return x.to(torch.bfloat16), gamma.to(torch.bfloat16)


# ------------------------------------------------------------- paged KV + attention

@dataclass
class PagedInputs:
    q: torch.Tensor            # [T, Hq, D] bf16, T = sum of q_lens
    k_new: torch.Tensor        # [T, Hkv, D] bf16 (the block's own keys)
    v_new: torch.Tensor        # [T, Hkv, D] bf16
    k_cache: torch.Tensor      # [num_pages, Hkv, PAGE, D] bf16
    v_cache: torch.Tensor      # [num_pages, Hkv, PAGE, D] bf16
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32, includes the new tokens
    cu_q: torch.Tensor         # [B+1] int32
    page_size: int

    @property
    def B(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def T(self) -> int:
        return int(self.q.shape[0])


def paged_inputs(seq_lens, q_lens, Hq: int, Hkv: int, D: int, seed: int,
                 page_size: int = PAGE_SIZE, spare_pages: int = 3, kv_std: float = 1.0,
                 q_std: float = 1.0, device: str = "cpu") -> PagedInputs:
    """A batch of sequences whose caches hold seq_lens[b] tokens (the last q_lens[b] of
    them being the verify block's own tokens, delivered separately in k_new/v_new).
    Every page of the pool is filled with N(0, kv_std) so slots nobody owns are finite;
    physical pages are handed out in a seeded random order.  ``device='cuda'`` draws the
    large cache tensors with the CUDA generator (same recipe, different stream)."""
    seq_lens = [int(s) for s in seq_lens]
    q_lens = [int(q) for q in q_lens]
    if len(seq_lens) != len(q_lens):
        raise ValueError("seq_lens and q_lens differ in length")
    for s, ql in zip(seq_lens, q_lens):
        if ql < 0 or s < ql:
            raise ValueError("each sequence must hold at least its block")
    B = len(seq_lens)
    g = generator(seed)
    pages_per_seq = [max(1, -(-s // page_size)) for s in seq_lens]
    max_pages = max(pages_per_seq) if B else 1
    num_pages = sum(pages_per_seq) + spare_pages
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    block_table = torch.full((max(B, 1), max_pages), -1, dtype=torch.int32)[:B]
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        block_table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    T = sum(q_lens)
    cu = [0]
    for ql in q_lens:
        cu.append(cu[-1] + ql)
    shape = (num_pages, Hkv, page_size, D)
    if device == "cpu":
        k_cache = (torch.randn(*shape, generator=g) * kv_std).to(torch.bfloat16)
        v_cache = (torch.randn(*shape, generator=g) * kv_std).to(torch.bfloat16)
    else:
        gc = torch.Generator(device=device)
        gc.manual_seed(int(seed) + 17)
        k_cache = (torch.randn(*shape, generator=gc, device=device) * kv_std).to(torch.bfloat16)
        v_cache = (torch.randn(*shape, generator=gc, device=device) * kv_std).to(torch.bfloat16)
    q = (torch.randn(T, Hq, D, generator=g) * q_std).to(torch.bfloat16)
    k_new = (torch.randn(T, Hkv, D, generator=g) * kv_std).to(torch.bfloat16)
    v_new = (torch.randn(T, Hkv, D, generator=g) * kv_std).to(torch.bfloat16)
    return PagedInputs(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                       block_table=block_table.contiguous(),
                       seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                       cu_q=torch.tensor(cu, dtype=torch.int32), page_size=page_size)


def mixed_lengths(B: int, seed: int, choices=(1028, 8196, 16388, 65540)):
    """Sequence lengths drawn uniformly (seeded) from the pages' Lk values."""
    idx = torch.randint(0, len(choices), (B,), generator=generator(seed))
    return [int(choices[i]) for i in idx]


# --------------------------------------------------------- greedy-trace decoder stack

@dataclass(frozen=True)
class DecoderConfig:
    """Shape of a Llama-style decoder stack (sizes only)."""
    hidden: int
    heads: int
    kv_heads: int
    head_dim: int
    inter: int
    layers: int
    vocab: int
    context: int          # tokens already in every sequence's KV cache
    eps: float = 1e-5
    theta: float = 500000.0


# The full-decoder workload: Llama-3-8B shapes, 8 layers, 8192-token contexts.  The pages
# name no vocabulary size; 128256 is Llama-3's.
LLAMA3_8B_8L = DecoderConfig(hidden=4096, heads=32, kv_heads=8, head_dim=128, inter=14336,
                             layers=8, vocab=128256, context=8192)

# A stack the oracle runs in seconds: two layers, GQA with 2 query heads per KV head.
TINY_DECODER = DecoderConfig(hidden=256, heads=4, kv_heads=2, head_dim=64, inter=512,
                             layers=2, vocab=1000, context=100)


def _name_seed(seed: int, name: str) -> int:
    import zlib
    return (int(seed) * 1000003 + zlib.crc32(name.encode())) & 0x7fffffffffff


def _normal_on(shape, std: float, mean: float, seed: int, device) -> torch.Tensor:
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    return (t * std + mean).to(torch.bfloat16)


def decoder_weight_shapes(cfg: DecoderConfig) -> dict:
    """Every weight of the stack with its shape (nn.Linear matrices are [out, in])."""
    q, kv = cfg.heads * cfg.head_dim, cfg.kv_heads * cfg.head_dim
    shapes = {"embed": (cfg.vocab, cfg.hidden), "lm_head": (cfg.vocab, cfg.hidden),
              "final_norm": (cfg.hidden,)}
    for i in range(cfg.layers):
        p = f"l{i}."
        shapes.update({p + "attn_norm": (cfg.hidden,), p + "wq": (q, cfg.hidden),
                       p + "wk": (kv, cfg.hidden), p + "wv": (kv, cfg.hidden),
                       p + "wo": (cfg.hidden, q), p + "mlp_norm": (cfg.hidden,),
                       p + "w_gate": (cfg.inter, cfg.hidden), p + "w_up": (cfg.inter, cfg.hidden),
                       p + "w_down": (cfg.hidden, cfg.inter)})
    return shapes


def decoder_weights(cfg: DecoderConfig, seed: int, device="cpu", std: float = 0.02,
                    norm_std: float = 0.0) -> dict:
    """Random-init bf16 weights: matrices N(0, std); norm gains N(1, norm_std) (ones at
    the default 0, the usual initialisation).  Each tensor has its own seed, derived from
    its name, so a tensor does not depend on which others are drawn."""
    out = {}
    for name, shape in decoder_weight_shapes(cfg).items():
        if len(shape) == 1:
            out[name] = _normal_on(shape, norm_std, 1.0, _name_seed(seed, name), device)
        else:
            out[name] = _normal_on(shape, std, 0.0, _name_seed(seed, name), device)
    return out


def decoder_context(cfg: DecoderConfig, seq_id: int, layer: int, seed: int, device="cpu"):
    """K and V rows (bf16 [context, Hkv, D], N(0,1)) that stand for sequence seq_id's
    already-processed context in one layer.  They depend only on (seed, seq_id, layer),
    never on the batch the sequence is decoded in."""
    shape = (cfg.context, cfg.kv_heads, cfg.head_dim)
    base = _name_seed(seed, f"ctx.{seq_id}.{layer}")
    return (_normal_on(shape, 1.0, 0.0, base * 2 + 1, device),
            _normal_on(shape, 1.0, 0.0, base * 2 + 2, device))


def decoder_first_token(cfg: DecoderConfig, seq_id: int, seed: int) -> int:
    """The token sequence seq_id is decoded from (uniform over the vocabulary)."""
    g = generator(_name_seed(seed, f"tok.{seq_id}"))
    return int(torch.randint(0, cfg.vocab, (1,), generator=g).item())


def decoder_prompt(cfg: DecoderConfig, seq_id: int, seed: int, length: int) -> list:
    """Sequence seq_id's prompt: `length` token ids, uniform over the vocabulary."""
    g = generator(_name_seed(seed, f"prompt.{seq_id}"))
    return torch.randint(0, cfg.vocab, (length,), generator=g).tolist()


def page_permutation(num_pages: int, seed: int) -> torch.Tensor:
    """A seeded permutation of physical page ids (int32)."""
    return torch.randperm(num_pages, generator=generator(seed)).to(torch.int32)


# ------------------------------------------------------------------ quantized weights

Q_MXFP4, Q_NVFP4, Q_MXFP8, Q_AFFINE4, Q_AFFINE8 = range(5)
Q_NAMES = {"mxfp4": Q_MXFP4, "nvfp4": Q_NVFP4, "mxfp8": Q_MXFP8, "affine4": Q_AFFINE4,
           "affine8": Q_AFFINE8}


def quant_weights(fmt: int, N: int, K: int, gs: int, seed: int, row_pad_bytes: int = 16):
    """Random codes and scales of a quantized W (no quantization arithmetic: the codes are
    drawn directly).  Returns (wq uint8 [N, row bytes], scales, biases or None); rows of wq
    are padded to a multiple of row_pad_bytes.  Block scales are E8M0 exponents near 2^-3
    (mx formats) or E4M3 codes of moderate positive values (nvfp4); affine scales are
    bf16 N(0, 0.005), biases bf16 N(0, 0.01).  FP8 codes avoid the NaN patterns."""
    g = generator(seed)
    four = fmt in (Q_MXFP4, Q_NVFP4, Q_AFFINE4)
    nbytes = K // 2 if four else K
    row = -(-nbytes // row_pad_bytes) * row_pad_bytes
    wq = torch.zeros(N, row, dtype=torch.uint8)
    codes = torch.randint(0, 256, (N, nbytes), generator=g, dtype=torch.int32)
    if fmt == Q_MXFP8:
        codes = torch.where((codes & 0x7F) == 0x7F, codes - 1, codes)  # no NaN codes
    wq[:, :nbytes] = codes.to(torch.uint8)
    groups = K // gs
    if fmt in (Q_MXFP4, Q_MXFP8):
        scales = torch.randint(120, 127, (N, groups), generator=g, dtype=torch.int32).to(torch.uint8)
        biases = None
    elif fmt == Q_NVFP4:
        scales = torch.randint(0x28, 0x40, (N, groups), generator=g, dtype=torch.int32).to(torch.uint8)
        biases = None
    else:
        scales = normal_bf16((N, groups), 0.0, 0.005, seed=seed * 7 + 1)
        biases = normal_bf16((N, groups), 0.0, 0.01, seed=seed * 7 + 2)
    return wq, scales, biases
