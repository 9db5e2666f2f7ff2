"""ctypes front end of the plain C oracle (``bi_oracle.c``).

TEST INFRASTRUCTURE ONLY: the product library never imports this package.  Only the
test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA path; inputs arrive as numpy arrays of bf16 bit
patterns (``uint16``) and results leave as unrounded fp32 plus, on request, the
oracle's own bf16 rounding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bi_oracle.c")
_LIB = os.path.join(_HERE, "libbi_oracle.so")

# Strict IEEE fp32: no fused multiply-add contraction, no fast-math reassociation.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (seconds); returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def _declare(L: ctypes.CDLL) -> None:
    L.oracle_bf16_round.argtypes = [_p, _p, _i64]
    L.oracle_bf16_widen.argtypes = [_p, _p, _i64]
    L.oracle_left_fold_f64.argtypes = [_p, _i64]
    L.oracle_left_fold_f64.restype = ctypes.c_double
    for name in ("oracle_sum_sequential_f32", "oracle_sum_pairwise_f32", "oracle_sum_squares_f32"):
        getattr(L, name).argtypes = [_p, _i64]
        getattr(L, name).restype = ctypes.c_float
    L.oracle_sum_split_f32.argtypes = [_p, _i64, _i64]
    L.oracle_sum_split_f32.restype = ctypes.c_float
    L.oracle_argmax_f32.argtypes = [_p, _i64]
    L.oracle_argmax_f32.restype = _i64
    L.oracle_matmul.argtypes = [_p, _i64, _p, _i64, ctypes.c_int, _p, _i64, _i64, _i64, _i64]
    L.oracle_rmsnorm.argtypes = [_p, _i64, _p, _p, _i64, _i64, _i64, ctypes.c_float]
    L.oracle_kv_append.argtypes = [_p, _p, _p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64]
    L.oracle_attention_row.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64,
                                       _i64, _i64, _i64, ctypes.c_float, _p, _p]
    L.oracle_attention_row.restype = ctypes.c_int
    L.oracle_attention.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.c_float, _p, _p]
    L.oracle_attention.restype = ctypes.c_int
    L.oracle_positions.argtypes = [_p, _p, _i64, _p]
    L.oracle_rope.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _i64, _p, ctypes.c_double]
    L.oracle_swiglu.argtypes = [_p, _p, _p, _i64]
    L.oracle_add.argtypes = [_p, _p, _p, _i64]
    L.oracle_log_softmax_f32.argtypes = [_p, _i64, _p, _i64, _i64, _i64]
    L.oracle_f16_widen.argtypes = [_p, _p, _i64]
    for name in ("oracle_decode_fp4", "oracle_decode_fp8", "oracle_decode_e8m0"):
        getattr(L, name).argtypes = [_p, _p, _i64]
    L.oracle_dequantize.argtypes = [_p, _i64, _p, _i64, _p, _i64, ctypes.c_int, _i64, _p, _i64,
                                    _i64]
    L.oracle_matmul_f32.argtypes = [_p, _i64, _p, _i64, ctypes.c_int, _p, _i64, _i64, _i64,
                                    _i64]
    L.oracle_rmsnorm_f32.argtypes = [_p, _i64, _p, _p, _i64, _i64, _i64, ctypes.c_float]
    L.oracle_matmul16.argtypes = [_p, _i64, _p, _i64, ctypes.c_int, _p, _i64, _i64, _i64, _i64,
                                  ctypes.c_int]
    L.oracle_rmsnorm16.argtypes = [_p, _i64, _p, _p, _i64, _i64, _i64, ctypes.c_float,
                                   ctypes.c_int]
    L.oracle_mean_f32.argtypes = [_p, _i64, _i64, _i64, _p]
    L.oracle_mean_bf16.argtypes = [_p, _i64, _i64, _i64, _p]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"oracle expects {np.dtype(dtype)}, got {a.dtype}")
    return a


# ----------------------------------------------------------------------------- bf16

def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = _as(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_bf16_round(_ptr(x), _ptr(out), x.size)
    return out


def bf16_widen(h: np.ndarray) -> np.ndarray:
    h = _as(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().oracle_bf16_widen(_ptr(h), _ptr(out), h.size)
    return out


# ------------------------------------------------------------------ reduction trees

def left_fold_f64(xs) -> float:
    a = _as(np.asarray(xs, dtype=np.float64), np.float64)
    return float(lib().oracle_left_fold_f64(_ptr(a), a.size))


def sum_sequential_f32(a) -> np.float32:
    a = _as(a, np.float32)
    return np.float32(lib().oracle_sum_sequential_f32(_ptr(a), a.size))


def sum_pairwise_f32(a) -> np.float32:
    a = _as(a, np.float32)
    return np.float32(lib().oracle_sum_pairwise_f32(_ptr(a), a.size))


def sum_split_f32(a, splits: int) -> np.float32:
    a = _as(a, np.float32)
    return np.float32(lib().oracle_sum_split_f32(_ptr(a), a.size, splits))


def sum_squares_f32(a) -> np.float32:
    a = _as(a, np.float32)
    return np.float32(lib().oracle_sum_squares_f32(_ptr(a), a.size))


def argmax_f32(v) -> int:
    v = _as(v, np.float32)
    return int(lib().oracle_argmax_f32(_ptr(v), v.size))


# --------------------------------------------------------------------------- matmul

W_NK, W_KN = 0, 1


def matmul(x: np.ndarray, w: np.ndarray, w_layout: int) -> np.ndarray:
    """x uint16 [M,K] (bf16 bits); w uint16 [N,K] (W_NK) or [K,N] (W_KN) -> fp32 [M,N]."""
    x = _as(x, np.uint16)
    w = _as(w, np.uint16)
    M, K = x.shape
    N = w.shape[0] if w_layout == W_NK else w.shape[1]
    Kw = w.shape[1] if w_layout == W_NK else w.shape[0]
    if Kw != K:
        raise ValueError("inner dimensions differ")
    y = np.empty((M, N), dtype=np.float32)
    lib().oracle_matmul(_ptr(x), K, _ptr(w), w.shape[1], w_layout, _ptr(y), N, M, N, K)
    return y


def matmul_strided(x, ldx, w, ldw, w_layout, M, N, K, ldy) -> np.ndarray:
    """Raw strided call: x, w flat uint16 buffers; returns flat fp32 [M*ldy]."""
    x = _as(x, np.uint16)
    w = _as(w, np.uint16)
    y = np.full(M * ldy, np.nan, dtype=np.float32)
    lib().oracle_matmul(_ptr(x), ldx, _ptr(w), ldw, w_layout, _ptr(y), ldy, M, N, K)
    return y


# -------------------------------------------------------------------------- rmsnorm

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x uint16 [rows,H], gamma uint16 [H] -> fp32 [rows,H] (unrounded)."""
    x = _as(x, np.uint16)
    gamma = _as(gamma, np.uint16)
    rows, H = x.shape
    y = np.empty((rows, H), dtype=np.float32)
    lib().oracle_rmsnorm(_ptr(x), H, _ptr(gamma), _ptr(y), H, rows, H, ctypes.c_float(eps))
    return y


# ----------------------------------------------------------------- paged attention

def kv_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens, cu_q, page_size):
    """Returns updated copies of (k_cache, v_cache) (uint16 [pages,Hkv,page,D])."""
    k_new = _as(k_new, np.uint16)
    v_new = _as(v_new, np.uint16)
    kc = _as(k_cache, np.uint16).copy()
    vc = _as(v_cache, np.uint16).copy()
    bt = _as(block_table, np.int32)
    sl = _as(seq_lens, np.int32)
    cq = _as(cu_q, np.int32)
    B = sl.size
    Hkv, D = kc.shape[1], kc.shape[3]
    lib().oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                           _ptr(sl), _ptr(cq), B, Hkv, D, page_size)
    return kc, vc


def attention(q, k_cache, v_cache, block_table, seq_lens, cu_q, Hq, scale):
    """q uint16 [T,Hq,D]; caches uint16 [pages,Hkv,page,D] -> (out fp32 [T,Hq,D], lse fp32 [T,Hq])."""
    q = _as(q, np.uint16)
    kc = _as(k_cache, np.uint16)
    vc = _as(v_cache, np.uint16)
    bt = _as(block_table, np.int32)
    sl = _as(seq_lens, np.int32)
    cq = _as(cu_q, np.int32)
    T, _, D = q.shape
    Hkv, page = kc.shape[1], kc.shape[2]
    out = np.empty((T, Hq, D), dtype=np.float32)
    lse = np.empty((T, Hq), dtype=np.float32)
    rc = lib().oracle_attention(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl),
                                _ptr(cq), sl.size, Hq, Hkv, D, page, ctypes.c_float(scale),
                                _ptr(out), _ptr(lse))
    if rc:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    return out, lse


def attention_row(q, k_cache, v_cache, block_table, seq_lens, cu_q, b, j, h, Hq, scale):
    """One (sequence b, query j, head h) row: (out fp32 [D], lse)."""
    q = _as(q, np.uint16)
    kc = _as(k_cache, np.uint16)
    vc = _as(v_cache, np.uint16)
    bt = _as(block_table, np.int32)
    sl = _as(seq_lens, np.int32)
    cq = _as(cu_q, np.int32)
    D = q.shape[-1]
    Hkv, page = kc.shape[1], kc.shape[2]
    out = np.empty(D, dtype=np.float32)
    lse = np.empty(1, dtype=np.float32)
    rc = lib().oracle_attention_row(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl),
                                    _ptr(cq), b, j, Hq, Hkv, D, page, h, ctypes.c_float(scale),
                                    _ptr(out), _ptr(lse))
    if rc:
        raise RuntimeError(f"oracle_attention_row failed ({rc})")
    return out, float(lse[0])


# ------------------------------------------------------------------- decoder glue

def positions(seq_lens, cu_q=None) -> np.ndarray:
    """Position of every token of a ragged block (int32 [T]); cu_q None = one per sequence."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if cu_q is None:
        pos = np.empty(sl.size, dtype=np.int32)
        lib().oracle_positions(_ptr(sl), None, sl.size, _ptr(pos))
        return pos
    cq = np.ascontiguousarray(cu_q, dtype=np.int32)
    pos = np.empty(int(cq[-1]), dtype=np.int32)
    lib().oracle_positions(_ptr(sl), _ptr(cq), sl.size, _ptr(pos))
    return pos


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """x uint16 [T,H,D] (bf16 bits), pos int32 [T] -> rotated fp64 [T,H,D] (unrounded)."""
    x = _as(x, np.uint16)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    T, H, D = x.shape
    if pos.size != T or D % 2:
        raise ValueError("pos must have one entry per token and D must be even")
    y = np.empty((T, H, D), dtype=np.float64)
    lib().oracle_rope(_ptr(x), H * D, _ptr(y), H * D, T, H, D, _ptr(pos), float(theta))
    return y


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u elementwise for bf16 bits g, u (same shape) -> fp64 (unrounded)."""
    g = _as(g, np.uint16)
    u = _as(u, np.uint16)
    if g.shape != u.shape:
        raise ValueError("g and u shapes differ")
    y = np.empty(g.shape, dtype=np.float64)
    lib().oracle_swiglu(_ptr(g), _ptr(u), _ptr(y), g.size)
    return y


def add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a + b elementwise for bf16 bits a, b (same shape) -> fp64 (exact)."""
    a = _as(a, np.uint16)
    b = _as(b, np.uint16)
    if a.shape != b.shape:
        raise ValueError("a and b shapes differ")
    y = np.empty(a.shape, dtype=np.float64)
    lib().oracle_add(_ptr(a), _ptr(b), _ptr(y), a.size)
    return y


BF16, F16 = 0, 2  # 16-bit input types of matmul16 / rmsnorm16


def f16_widen(h: np.ndarray) -> np.ndarray:
    """binary16 bit patterns -> fp32 values (exact), from the format definition."""
    h = _as(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().oracle_f16_widen(_ptr(h), _ptr(out), h.size)
    return out


def matmul16(x: np.ndarray, w: np.ndarray, w_layout: int, dtype: int) -> np.ndarray:
    """matmul for 16-bit bits of type dtype (BF16 or F16) -> unrounded fp32 [M, N]."""
    x = _as(x, np.uint16)
    w = _as(w, np.uint16)
    M, K = x.shape
    N = w.shape[0] if w_layout == W_NK else w.shape[1]
    y = np.empty((M, N), dtype=np.float32)
    lib().oracle_matmul16(_ptr(x), K, _ptr(w), w.shape[1], w_layout, _ptr(y), N, M, N, K,
                          int(dtype))
    return y


def rmsnorm16(x: np.ndarray, gamma: np.ndarray, eps: float, dtype: int) -> np.ndarray:
    """RMSNorm for 16-bit bits of type dtype (BF16 or F16) -> unrounded fp32 [rows, H]."""
    x = _as(x, np.uint16)
    gamma = _as(gamma, np.uint16)
    rows, H = x.shape
    y = np.empty((rows, H), dtype=np.float32)
    lib().oracle_rmsnorm16(_ptr(x), H, _ptr(gamma), _ptr(y), H, rows, H, float(eps), int(dtype))
    return y


def matmul_f32(x: np.ndarray, w: np.ndarray, w_layout: int) -> np.ndarray:
    """matmul of fp32 x [M, K] and w (NK [N, K] or KN [K, N]) -> fp64 (exact products,
    fp64 sum)."""
    x = _as(x, np.float32)
    w = _as(w, np.float32)
    M, K = x.shape
    N = w.shape[0] if w_layout == W_NK else w.shape[1]
    y = np.empty((M, N), dtype=np.float64)
    lib().oracle_matmul_f32(_ptr(x), K, _ptr(w), w.shape[1], w_layout, _ptr(y), N, M, N, K)
    return y


def rmsnorm_f32(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of fp32 [rows, H] with fp32 gamma, the book's fp32 procedure."""
    x = _as(x, np.float32)
    gamma = _as(gamma, np.float32)
    rows, H = x.shape
    y = np.empty((rows, H), dtype=np.float32)
    lib().oracle_rmsnorm_f32(_ptr(x), H, _ptr(gamma), _ptr(y), H, rows, H, float(eps))
    return y


# quantized weight formats (the encodings are documented in bi_oracle.c)
Q_MXFP4, Q_NVFP4, Q_MXFP8, Q_AFFINE4, Q_AFFINE8 = range(5)


def _decode(fn, codes):
    codes = _as(codes, np.uint8)
    out = np.empty(codes.shape, dtype=np.float32)
    fn(_ptr(codes), _ptr(out), codes.size)
    return out


def decode_fp4(codes):
    """FP4 E2M1 codes (low 4 bits of each byte) -> fp32 values."""
    return _decode(lib().oracle_decode_fp4, codes)


def decode_fp8(codes):
    """FP8 E4M3 codes -> fp32 values (0x7F / 0xFF are NaN; no infinities)."""
    return _decode(lib().oracle_decode_fp8, codes)


def decode_e8m0(codes):
    """E8M0 scale codes -> 2^(code-127) (255 is NaN)."""
    return _decode(lib().oracle_decode_e8m0, codes)


def dequantize(wq, scales, biases, fmt: int, gs: int, N: int, K: int) -> np.ndarray:
    """Quantized W (NK: one row per output column) -> bf16 bits [N, K].  wq: uint8 codes
    [N, K/2] (4-bit, low nibble first) or [N, K] (8-bit); scales: uint8 [N, K/gs] (block
    formats) or bf16 bits [N, K/gs] (affine, with biases the same)."""
    wq = _as(wq, np.uint8)
    affine = fmt in (Q_AFFINE4, Q_AFFINE8)
    scales = _as(scales, np.uint16 if affine else np.uint8)
    b = _as(biases, np.uint16) if affine else np.zeros((1, 1), dtype=np.uint16)
    out = np.empty((N, K), dtype=np.uint16)
    lib().oracle_dequantize(_ptr(wq), wq.shape[1], _ptr(scales), scales.shape[1], _ptr(b),
                            b.shape[1], int(fmt), int(gs), _ptr(out), N, K)
    return out


def qmatmul(x: np.ndarray, wq, scales, biases, fmt: int, gs: int, N: int) -> np.ndarray:
    """bf16 x [M, K] times dequantized W^T -> unrounded fp32 [M, N] (the matmul above)."""
    x = _as(x, np.uint16)
    return matmul(x, dequantize(wq, scales, biases, fmt, gs, N, x.shape[1]), W_NK)


def log_softmax(x: np.ndarray) -> np.ndarray:
    """Row-wise log-softmax of fp32 [rows, n] (or [n]) -> fp64, by the definition."""
    x = _as(x, np.float32)
    x2 = x.reshape(1, -1) if x.ndim == 1 else x
    rows, n = x2.shape
    y = np.empty((rows, n), dtype=np.float64)
    lib().oracle_log_softmax_f32(_ptr(x2), n, _ptr(y), n, rows, n)
    return y.reshape(x.shape)


def mean(x: np.ndarray, bf16: bool = False) -> np.ndarray:
    """Row means of [rows, n] (fp32 values, or bf16 bits with bf16=True) -> fp64 [rows]."""
    x = _as(x, np.uint16 if bf16 else np.float32)
    x2 = x.reshape(1, -1) if x.ndim == 1 else x
    rows, n = x2.shape
    out = np.empty(rows, dtype=np.float64)
    fn = lib().oracle_mean_bf16 if bf16 else lib().oracle_mean_f32
    fn(_ptr(x2), n, rows, n, _ptr(out))
    return out


def to_bf16(y: np.ndarray) -> np.ndarray:
    """Unrounded oracle values (fp32 or fp64) -> bf16 bits: fp64 narrows to fp32 (round
    to nearest even), then fp32 rounds to bf16 (nearest even)."""
    return bf16_round(np.asarray(y, dtype=np.float32))
