"""Batch-invariant transformer reductions for one NVIDIA GB300 (sm_103a).

The compute lives in ``libbi.so`` -- hand-written CUDA kernels behind the C ABI declared
in ``include/bi.h``.  This module is its thin ctypes binding: it checks that tensors are
CUDA tensors of the right dtype, reads their pointers, strides and the current stream,
and calls the C entry point of the same name.  Outputs it is asked to create are
allocated with torch (device memory is torch's job); every arithmetic step runs in the
kernels.  There is no CPU fallback: if the library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("BI_LIBRARY_PATH") or os.path.join(HERE, "libbi.so")

BI_OK, BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED, BI_ERR_CUDA, BI_ERR_TIMEOUT, BI_ERR_DEVICE_ARG = range(6)
BI_BF16, BI_F32, BI_F16 = 0, 1, 2
BI_W_NK, BI_W_KN = 0, 1
PAGE_SIZE = 64
ATTN_CHUNK = 512
ATTN_MAX_Q = 8
ATTN_MAX_ROWS = 32
STATIC_WS_BYTES = 32 * 1024 * 1024

# every function include/bi.h, include/bi_glue.h and include/bi_rowwise.h declare, with
# its ctypes signature
_p, _i64, _f32, _sz, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "bi_abi_version": ([], _int),
    "bi_status_string": ([_int], ctypes.c_char_p),
    "bi_last_error_message": ([], ctypes.c_char_p),
    "bi_set_batch_invariant_limit": ([_i64], _int),
    "bi_get_batch_invariant_limit": ([], _i64),
    "bi_within_batch_invariant_limit": ([_i64], _int),
    "bi_set_weight_prefetch": ([_int], _int),
    "bi_get_weight_prefetch": ([], _int),
    "bi_matmul_splits": ([_i64, _i64, _i64, _int, _int], _int),
    "bi_attn_chunk": ([_i64, _i64, _i64, _i64, _i64, _i64, _i64, _sz, _int], _i64),
    "bi_matmul": ([_p, _i64, _p, _i64, _int, _p, _i64, _int, _i64, _i64, _i64, _p], _int),
    "bi_matmul_ex": ([_p, _i64, _p, _i64, _int, _p, _i64, _int, _int, _i64, _i64, _i64, _p],
                     _int),
    "bi_qmatmul": ([_p, _i64, _p, _i64, _p, _i64, _p, _i64, _int, _int, _p, _i64, _int, _i64,
                    _i64, _i64, _p], _int),
    "bi_qmatmul_ex": ([_p, _i64, _p, _i64, _p, _i64, _p, _i64, _int, _int, _int, _p, _i64, _int,
                       _i64, _i64, _i64, _p], _int),
    "bi_rmsnorm": ([_p, _i64, _p, _p, _i64, _int, _i64, _i64, _f32, _p], _int),
    "bi_rmsnorm_ex": ([_p, _i64, _p, _p, _i64, _int, _int, _i64, _i64, _f32, _p], _int),
    "bi_kv_append": ([_p, _p, _p, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64, _p],
                     _int),
    "bi_attn_workspace_size": ([_i64, _i64, _i64, _i64], _sz),
    "bi_verify_block": ([_p, _p, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                         _i64, _i64, _f32, _p, _p, _p, _sz, _p], _int),
    "bi_prefill_attn": ([_p, _p, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                         _i64, _i64, _f32, _p, _p, _p, _sz, _p], _int),
    "bi_decode_attn": ([_p, _p, _p, _i64, _p, _i64, _p, _i64, _i64, _i64, _i64, _i64, _i64, _f32,
                        _p, _p, _p, _sz, _p], _int),
    "bi_verify_block_static_ws": ([_p, _p, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _i64,
                                   _i64, _i64, _i64, _f32, _p, _p, _p], _int),
    "bi_device_status": ([_p], _int),
    "bi_selftest_wait_timeout": ([ctypes.c_uint64, _p], _int),
    "bi_selftest_set_wait_budget": ([ctypes.c_uint64, _p], _int),
    # decoder glue (include/bi_glue.h)
    "bi_embedding": ([_p, _i64, _i64, _p, _i64, _p, _i64, _p], _int),
    "bi_rope": ([_p, _i64, _i64, _i64, _i64, _p, _p, _i64, _f32, _p], _int),
    "bi_swiglu": ([_p, _i64, _p, _i64, _p, _i64, _i64, _i64, _p], _int),
    "bi_add": ([_p, _p, _p, _i64, _p], _int),
    "bi_argmax": ([_p, _i64, _i64, _i64, _p, _p], _int),
    # row-wise reductions (include/bi_rowwise.h)
    "bi_log_softmax": ([_p, _i64, _p, _i64, _i64, _i64, _p], _int),
    "bi_mean": ([_p, _i64, _int, _i64, _i64, _p, _p], _int),
}

_lib: Optional[ctypes.CDLL] = None


class BIError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def _status_name(s: int) -> str:
    names = ["BI_OK", "BI_ERR_INVALID_ARG", "BI_ERR_UNSUPPORTED", "BI_ERR_CUDA", "BI_ERR_TIMEOUT",
             "BI_ERR_DEVICE_ARG"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def lib() -> ctypes.CDLL:
    """The loaded libbi.so (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbi.so not found at {LIB_PATH}; build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != BI_OK:
        msg = lib().bi_last_error_message().decode(errors="replace")
        raise BIError(status, msg)


def _torch():
    import torch
    return torch


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, dtype, name, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")


def _row_major_2d(t, name):
    if t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


# ------------------------------------------------------------------------------ limit

def set_batch_invariant_limit(limit: int) -> None:
    _check(lib().bi_set_batch_invariant_limit(int(limit)))


def get_batch_invariant_limit() -> int:
    return int(lib().bi_get_batch_invariant_limit())


def within_batch_invariant_limit(dim: int) -> bool:
    return bool(lib().bi_within_batch_invariant_limit(int(dim)))


def set_weight_prefetch(on: bool) -> None:
    """Let matmuls start reading their weights before the previous kernel in the stream
    has finished.  Only for weights no kernel writes right before the call reads them."""
    _check(lib().bi_set_weight_prefetch(1 if on else 0))


def get_weight_prefetch() -> bool:
    return bool(lib().bi_get_weight_prefetch())


def matmul_splits(M: int, N: int, K: int, w_layout: str = "nk", num_sms: int = 152) -> int:
    """How many CTAs would share each output tile's K range for this shape under the
    current limit (1: the invariant K loop).  0 for invalid sizes."""
    lay = {"nk": BI_W_NK, "kn": BI_W_KN}[w_layout]
    return int(lib().bi_matmul_splits(int(M), int(N), int(K), lay, int(num_sms)))


def attn_chunk(batch: int, total_q: int, max_q: int, max_seq_len: int, num_q_heads: int,
               num_kv_heads: int, head_dim: int, workspace_bytes: int,
               num_sms: int = 152) -> int:
    """The split-KV chunk length (keys) a verify/decode call with these sizes would use
    under the current limit (ATTN_CHUNK inside it).  0 for invalid sizes."""
    return int(lib().bi_attn_chunk(int(batch), int(total_q), int(max_q), int(max_seq_len),
                                   int(num_q_heads), int(num_kv_heads), int(head_dim),
                                   int(workspace_bytes), int(num_sms)))


# ----------------------------------------------------------------------------- matmul

def _in_dtype(t, name):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BI_BF16
    if t.dtype == torch.float16:
        return BI_F16
    if t.dtype == torch.float32:
        return BI_F32
    raise ValueError(f"{name} must be bf16, fp16 or fp32")


def matmul(x, w, w_layout: str = "nk", out=None, out_dtype=None, stream=None):
    """Y = X @ W for X [M,K] and W [N,K] ("nk", nn.Linear) or [K,N] ("kn"), both bf16, both
    fp16 or both fp32; Y in the input type or fp32."""
    torch = _torch()
    dt = _in_dtype(x, "x")
    _need(x, x.dtype, "x", 2)
    _need(w, x.dtype, "w", 2)
    layout = {"nk": BI_W_NK, "kn": BI_W_KN}[w_layout]
    M, K = x.shape
    N = w.shape[0] if layout == BI_W_NK else w.shape[1]
    if (w.shape[1] if layout == BI_W_NK else w.shape[0]) != K:
        raise ValueError("inner dimensions of x and w differ")
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype or x.dtype, device=x.device)
    if out.dtype not in (x.dtype, torch.float32) or tuple(out.shape) != (M, N):
        raise ValueError("out must be [M,N] of the input type or fp32")
    _check(lib().bi_matmul_ex(_ptr(x), _row_major_2d(x, "x"), _ptr(w), _row_major_2d(w, "w"),
                              layout, _ptr(out), _row_major_2d(out, "out"), dt,
                              BI_F32 if out.dtype == torch.float32 else dt, M, N, K,
                              _stream(stream)))
    return out


# ------------------------------------------------------------------- quantized matmul

Q_FORMATS = {"mxfp4": 0, "nvfp4": 1, "mxfp8": 2, "affine4": 3, "affine8": 4}


def qmatmul(x, wq, scales, fmt: str, group_size: int, K: int, biases=None, out=None,
            out_dtype=None, stream=None, layout: str = "nk", N: Optional[int] = None):
    """Y = X @ dequant(W)^T for bf16 X [M, K] and quantized W: layout "nk" (uint8 codes
    [N, row bytes], quantized along K) or "kn" (codes [K, row bytes] quantized along N;
    N must be given); see include/bi.h for the encodings.  Y bf16 or fp32."""
    torch = _torch()
    q = Q_FORMATS[fmt]
    _need(x, torch.bfloat16, "x", 2)
    _need(wq, torch.uint8, "wq", 2)
    M, kx = x.shape
    if kx != K:
        raise ValueError("x must have K columns")
    lay = {"nk": BI_W_NK, "kn": BI_W_KN}[layout]
    if lay == BI_W_NK:
        N = wq.shape[0]
    elif N is None or wq.shape[0] != K:
        raise ValueError("layout 'kn' needs N and codes [K, row bytes]")
    affine = fmt.startswith("affine")
    _need(scales, torch.bfloat16 if affine else torch.uint8, "scales", 2)
    if affine:
        _need(biases, torch.bfloat16, "biases", 2)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype or torch.bfloat16, device=x.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (M, N):
        raise ValueError("out must be [M,N] bf16 or fp32")
    _check(lib().bi_qmatmul_ex(
        _ptr(x), _row_major_2d(x, "x"), _ptr(wq), wq.stride(0), _ptr(scales), scales.stride(0),
        _ptr(biases) if affine else None, biases.stride(0) if affine else 0, q, int(group_size),
        lay, _ptr(out), _row_major_2d(out, "out"),
        BI_F32 if out.dtype == torch.float32 else BI_BF16, M, int(N), K, _stream(stream)))
    return out


# ---------------------------------------------------------------------------- rmsnorm

def rmsnorm(x, gamma, eps: float, out=None, out_dtype=None, stream=None):
    """y = x * rsqrt(mean(x^2) + eps) * gamma over the last dim of [rows, H] x; x and
    gamma both bf16, both fp16 or both fp32; y in the input type or fp32."""
    torch = _torch()
    dt = _in_dtype(x, "x")
    _need(x, x.dtype, "x", 2)
    _need(gamma, x.dtype, "gamma", 1)
    rows, H = x.shape
    if gamma.shape[0] != H or gamma.stride(0) != 1:
        raise ValueError("gamma must be a contiguous [H] tensor")
    if out is None:
        out = torch.empty(rows, H, dtype=out_dtype or x.dtype, device=x.device)
    if out.dtype not in (x.dtype, torch.float32):
        raise ValueError("out must be of the input type or fp32")
    _check(lib().bi_rmsnorm_ex(_ptr(x), _row_major_2d(x, "x"), _ptr(gamma), _ptr(out),
                               _row_major_2d(out, "out"), dt,
                               BI_F32 if out.dtype == torch.float32 else dt, rows, H,
                               float(eps), _stream(stream)))
    return out


# ------------------------------------------------------------------ paged attention

def _paged_common(k_cache, v_cache, block_table, seq_lens):
    torch = _torch()
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and block_table.is_contiguous()
            and seq_lens.is_contiguous()):
        raise ValueError("caches, block_table and seq_lens must be contiguous")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    num_pages, hkv, page, d = k_cache.shape
    return num_pages, hkv, page, d


def kv_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens, cu_q, stream=None):
    """Writes the block's new keys/values into their cache slots (before attention)."""
    torch = _torch()
    num_pages, hkv, page, d = _paged_common(k_cache, v_cache, block_table, seq_lens)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    if not (k_new.is_contiguous() and v_new.is_contiguous() and cu_q.is_contiguous()):
        raise ValueError("k_new, v_new and cu_q must be contiguous")
    B = seq_lens.shape[0]
    _check(lib().bi_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_pages,
                              _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(cu_q),
                              B, k_new.shape[0], hkv, d, page, _stream(stream)))


def attn_workspace_size(total_q: int, num_q_heads: int, head_dim: int, max_seq_len: int) -> int:
    return int(lib().bi_attn_workspace_size(total_q, num_q_heads, head_dim, max_seq_len))


def _attn_out(q, out, lse, want_lse):
    torch = _torch()
    T, hq, d = q.shape
    if out is None:
        out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out", 3)
    if not out.is_contiguous() or tuple(out.shape) != (T, hq, d):
        raise ValueError("out must be a contiguous [T, Hq, D] bf16 tensor")
    if lse is None and want_lse:
        lse = torch.empty(T, hq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse", 2)
        if not lse.is_contiguous() or tuple(lse.shape) != (T, hq):
            raise ValueError("lse must be a contiguous [T, Hq] fp32 tensor")
    return out, lse


def _workspace(workspace, need, device):
    torch = _torch()
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def verify_block(q, k_cache, v_cache, block_table, seq_lens, cu_q, max_q: int, max_seq_len: int,
                 scale: float, out=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Causal attention of each sequence's new block (q bf16 [T,Hq,D]) over its paged cache."""
    torch = _torch()
    num_pages, hkv, page, d = _paged_common(k_cache, v_cache, block_table, seq_lens)
    _need(q, torch.bfloat16, "q", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    if not q.is_contiguous() or not cu_q.is_contiguous():
        raise ValueError("q and cu_q must be contiguous")
    T, hq, _ = q.shape
    out, lse = _attn_out(q, out, lse, want_lse)
    ws, ws_bytes = _workspace(workspace, attn_workspace_size(T, hq, d, max_seq_len), q.device)
    _check(lib().bi_verify_block(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages,
                                 _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                 _ptr(cu_q), seq_lens.shape[0], T, int(max_q), int(max_seq_len),
                                 hq, hkv, d, page, float(scale), _ptr(out), _ptr(lse), _ptr(ws),
                                 ws_bytes, _stream(stream)))
    return out, lse


def prefill_attn(q, k_cache, v_cache, block_table, seq_lens, cu_q, max_q: int, max_seq_len: int,
                 scale: float, out=None, lse=None, want_lse=True, workspace=None, stream=None):
    """verify_block for blocks of any width (chunked prefill, prefix caching): every query
    reduced exactly as verify_block / decode_attn reduce it."""
    torch = _torch()
    num_pages, hkv, page, d = _paged_common(k_cache, v_cache, block_table, seq_lens)
    _need(q, torch.bfloat16, "q", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    if not q.is_contiguous() or not cu_q.is_contiguous():
        raise ValueError("q and cu_q must be contiguous")
    T, hq, _ = q.shape
    out, lse = _attn_out(q, out, lse, want_lse)
    ws, ws_bytes = _workspace(workspace, attn_workspace_size(T, hq, d, max_seq_len), q.device)
    _check(lib().bi_prefill_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages,
                                 _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                 _ptr(cu_q), seq_lens.shape[0], T, int(max_q), int(max_seq_len),
                                 hq, hkv, d, page, float(scale), _ptr(out), _ptr(lse), _ptr(ws),
                                 ws_bytes, _stream(stream)))
    return out, lse


def verify_block_static_ws(q, k_cache, v_cache, block_table, seq_lens, cu_q, max_q: int,
                           max_seq_len: int, scale: float, out=None, lse=None, want_lse=True,
                           stream=None):
    """verify_block with the library's fixed device workspace instead of one from the
    caller: for callers that cannot allocate device memory (see include/bi.h).  Calls
    whose kernels overlap on the GPU share that workspace and must not overlap."""
    torch = _torch()
    num_pages, hkv, page, d = _paged_common(k_cache, v_cache, block_table, seq_lens)
    _need(q, torch.bfloat16, "q", 3)
    _need(cu_q, torch.int32, "cu_q", 1)
    if not q.is_contiguous() or not cu_q.is_contiguous():
        raise ValueError("q and cu_q must be contiguous")
    T, hq, _ = q.shape
    out, lse = _attn_out(q, out, lse, want_lse)
    _check(lib().bi_verify_block_static_ws(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages,
                                           _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                           _ptr(cu_q), seq_lens.shape[0], T, int(max_q),
                                           int(max_seq_len), hq, hkv, d, page, float(scale),
                                           _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def decode_attn(q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                out=None, lse=None, want_lse=True, workspace=None, stream=None):
    """One new token per sequence: q bf16 [B,Hq,D]; token b is the last position of b."""
    torch = _torch()
    num_pages, hkv, page, d = _paged_common(k_cache, v_cache, block_table, seq_lens)
    _need(q, torch.bfloat16, "q", 3)
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    B, hq, _ = q.shape
    out, lse = _attn_out(q, out, lse, want_lse)
    ws, ws_bytes = _workspace(workspace, attn_workspace_size(B, hq, d, max_seq_len), q.device)
    _check(lib().bi_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages,
                                _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                int(max_seq_len), hq, hkv, d, page, float(scale), _ptr(out),
                                _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)))
    return out, lse


# ---------------------------------------------------------------------- device status

def device_status(stream=None) -> int:
    """Synchronises the stream; returns the bi_status of the device error word (and
    clears it)."""
    return int(lib().bi_device_status(_stream(stream)))


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib().bi_selftest_wait_timeout(int(timeout_ns), _stream(stream)))


def selftest_set_wait_budget(timeout_ns: int, stream=None) -> None:
    """Budget of every bounded wait in the kernels (ns; 0 = the library default).  Tests
    only: see include/bi.h."""
    _check(lib().bi_selftest_set_wait_budget(int(timeout_ns), _stream(stream)))


# ----------------------------------------------------------------------- decoder glue

def embedding(table, ids, out=None, stream=None):
    """out[t] = table[ids[t]] for a bf16 [vocab, hidden] table and int32 ids [n]."""
    torch = _torch()
    _need(table, torch.bfloat16, "table", 2)
    _need(ids, torch.int32, "ids", 1)
    if not table.is_contiguous() or not ids.is_contiguous():
        raise ValueError("table and ids must be contiguous")
    vocab, hidden = table.shape
    n = ids.shape[0]
    if out is None:
        out = torch.empty(n, hidden, dtype=torch.bfloat16, device=table.device)
    _need(out, torch.bfloat16, "out", 2)
    if tuple(out.shape) != (n, hidden):
        raise ValueError("out must be [n, hidden]")
    _check(lib().bi_embedding(_ptr(table), vocab, hidden, _ptr(ids), n, _ptr(out),
                              _row_major_2d(out, "out"), _stream(stream)))
    return out


def rope(x, seq_lens, cu_q=None, theta: float = 500000.0, stream=None):
    """Rotary embedding in place on x bf16 [T, H, D] (rows may be strided: x[t] at
    x.stride(0)); positions from seq_lens / cu_q as in verify_block."""
    torch = _torch()
    _need(x, torch.bfloat16, "x", 3)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    T, H, D = x.shape
    if x.stride(2) != 1 or x.stride(1) != D:
        raise ValueError("x must have contiguous heads within a token")
    if cu_q is not None:
        _need(cu_q, torch.int32, "cu_q", 1)
    _check(lib().bi_rope(_ptr(x), x.stride(0) if T > 1 else H * D, T, H, D, _ptr(seq_lens),
                         _ptr(cu_q), seq_lens.shape[0], float(theta), _stream(stream)))
    return x


def swiglu(gate, up, out=None, stream=None):
    """silu(gate) * up elementwise for bf16 [rows, inter] gate and up."""
    torch = _torch()
    _need(gate, torch.bfloat16, "gate", 2)
    _need(up, torch.bfloat16, "up", 2)
    if gate.shape != up.shape:
        raise ValueError("gate and up shapes differ")
    rows, inter = gate.shape
    if out is None:
        out = torch.empty(rows, inter, dtype=torch.bfloat16, device=gate.device)
    _need(out, torch.bfloat16, "out", 2)
    _check(lib().bi_swiglu(_ptr(gate), _row_major_2d(gate, "gate"), _ptr(up),
                           _row_major_2d(up, "up"), _ptr(out), _row_major_2d(out, "out"), rows,
                           inter, _stream(stream)))
    return out


def add(a, b, out=None, stream=None):
    """a + b elementwise for contiguous bf16 tensors of one shape (out may be a or b)."""
    torch = _torch()
    _need(a, torch.bfloat16, "a")
    _need(b, torch.bfloat16, "b")
    if a.shape != b.shape or not a.is_contiguous() or not b.is_contiguous():
        raise ValueError("a and b must be contiguous tensors of one shape")
    if out is None:
        out = torch.empty_like(a)
    _need(out, torch.bfloat16, "out")
    if out.shape != a.shape or not out.is_contiguous():
        raise ValueError("out must be contiguous with a's shape")
    _check(lib().bi_add(_ptr(a), _ptr(b), _ptr(out), a.numel(), _stream(stream)))
    return out


def argmax(logits, out=None, stream=None):
    """Greedy token of each row of fp32 [rows, n] logits (int32 [rows]); lowest index among
    equal maxima, NaN ranked below every number."""
    torch = _torch()
    _need(logits, torch.float32, "logits", 2)
    rows, n = logits.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    _need(out, torch.int32, "out", 1)
    if out.shape[0] != rows or not out.is_contiguous():
        raise ValueError("out must be a contiguous int32 [rows] tensor")
    _check(lib().bi_argmax(_ptr(logits), _row_major_2d(logits, "logits"), rows, n, _ptr(out),
                           _stream(stream)))
    return out


# ------------------------------------------------------------------ row-wise reductions

def log_softmax(x, out=None, stream=None):
    """Row-wise log-softmax of fp32 [rows, n] (one CTA per row, fixed tree); out may be x."""
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    rows, n = x.shape
    if out is None:
        out = torch.empty_like(x)
    _need(out, torch.float32, "out", 2)
    if tuple(out.shape) != (rows, n):
        raise ValueError("out must have the shape of x")
    _check(lib().bi_log_softmax(_ptr(x), _row_major_2d(x, "x"), _ptr(out),
                                _row_major_2d(out, "out"), rows, n, _stream(stream)))
    return out


def mean(x, out=None, stream=None):
    """Row means (fp32 [rows]) of bf16 or fp32 [rows, n] (one CTA per row, fixed tree)."""
    torch = _torch()
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    _need(x, x.dtype, "x", 2)
    rows, n = x.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _need(out, torch.float32, "out", 1)
    if out.shape[0] != rows or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 [rows] tensor")
    dt = BI_BF16 if x.dtype == torch.bfloat16 else BI_F32
    _check(lib().bi_mean(_ptr(x), _row_major_2d(x, "x"), dt, rows, n, _ptr(out),
                         _stream(stream)))
    return out
