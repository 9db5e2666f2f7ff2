"""The C ABI without a GPU: the library loads, exports every function include/bi.h
declares, rejects bad arguments before touching CUDA, and implements the process-wide
batch-invariant limit ("Fix/speculative shape invariance", ml-explore/mlx PR 4279,
section Changes: set/get_batch_invariant_limit, environment variable, default 0)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import invariant_bi_matmul_gb300 as bi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("bi.h", "bi_glue.h", "bi_rowwise.h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_header_is_checked():
    assert sorted(os.listdir(os.path.join(ROOT, "include"))) == sorted(
        os.path.basename(h) for h in HEADERS)


@pytest.fixture(scope="module")
def L():
    return bi.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("bi_matmul", "bi_rmsnorm", "bi_decode_attn", "bi_verify_block", "bi_kv_append",
                 "bi_embedding", "bi_rope", "bi_swiglu", "bi_add", "bi_argmax",
                 "bi_set_batch_invariant_limit", "bi_get_batch_invariant_limit",
                 "bi_attn_workspace_size", "bi_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported_and_bound(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} not exported by libbi.so"
        assert name in bi.SIGNATURES, f"{name} has no ctypes signature in the binding"
    assert set(bi.SIGNATURES) == set(declared_functions())
    assert L.bi_abi_version() == 1


def test_status_strings(L):
    for s in range(6):
        assert L.bi_status_string(s).decode().startswith("BI_")


def test_limit_set_get_and_reject_negative(L):
    old = L.bi_get_batch_invariant_limit()
    try:
        assert L.bi_set_batch_invariant_limit(8) == bi.BI_OK
        assert L.bi_get_batch_invariant_limit() == 8
        assert L.bi_within_batch_invariant_limit(8) == 1
        assert L.bi_within_batch_invariant_limit(9) == 0
        assert L.bi_set_batch_invariant_limit(-1) == bi.BI_ERR_INVALID_ARG
        assert L.bi_get_batch_invariant_limit() == 8          # unchanged
        assert L.bi_set_batch_invariant_limit(0) == bi.BI_OK
        assert L.bi_within_batch_invariant_limit(1) == 0      # 0 = disabled
    finally:
        L.bi_set_batch_invariant_limit(old)


def test_weight_prefetch_set_get_and_reject_other_values(L):
    old = L.bi_get_weight_prefetch()
    try:
        assert old == 0                                        # off unless asked for
        assert L.bi_set_weight_prefetch(1) == bi.BI_OK
        assert L.bi_get_weight_prefetch() == 1
        assert L.bi_set_weight_prefetch(2) == bi.BI_ERR_INVALID_ARG
        assert L.bi_get_weight_prefetch() == 1                 # unchanged
        assert L.bi_set_weight_prefetch(0) == bi.BI_OK
        assert L.bi_get_weight_prefetch() == 0
    finally:
        L.bi_set_weight_prefetch(old)


@pytest.mark.parametrize("env,want", [("12", 12), ("0", 0), ("-3", 0), ("abc", 0), (None, 0)])
def test_limit_initial_value_from_environment(env, want):
    code = ("import invariant_bi_matmul_gb300 as bi; "
            "print(bi.get_batch_invariant_limit())")
    e = dict(os.environ)
    e.pop("BI_BATCH_INVARIANT_LIMIT", None)
    if env is not None:
        e["BI_BATCH_INVARIANT_LIMIT"] = env
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=e, capture_output=True,
                         text=True, check=True)
    assert int(out.stdout.strip()) == want


def test_limit_is_atomic_under_threads(L):
    import threading
    old = L.bi_get_batch_invariant_limit()
    vals = [1, 2, 4, 8, 16]

    def worker(v):
        for _ in range(2000):
            L.bi_set_batch_invariant_limit(v)
            assert L.bi_get_batch_invariant_limit() in vals

    ts = [threading.Thread(target=worker, args=(v,)) for v in vals]
    [t.start() for t in ts]
    [t.join() for t in ts]
    assert L.bi_get_batch_invariant_limit() in vals
    L.bi_set_batch_invariant_limit(old)


def _err(L):
    return L.bi_last_error_message().decode()


def test_matmul_argument_errors_before_launch(L):
    d = ctypes.c_void_p(16)
    # negative sizes, bad enums, short leading dims, misalignment
    assert L.bi_matmul(d, 8, d, 8, 0, d, 8, 0, -1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(d, 8, d, 8, 7, d, 8, 0, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(d, 8, d, 8, 0, d, 8, 9, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(d, 4, d, 8, 0, d, 8, 0, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert "ldx" in _err(L)
    assert L.bi_matmul(d, 8, d, 4, 1, d, 8, 0, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(d, 8, d, 8, 0, d, 4, 0, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(None, 8, d, 8, 0, d, 8, 0, 1, 8, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_matmul(ctypes.c_void_p(18), 8, d, 8, 0, d, 8, 0, 1, 8, 8, None) == \
        bi.BI_ERR_UNSUPPORTED
    assert L.bi_matmul(d, 12, d, 16, 0, d, 8, 0, 1, 8, 12, None) == bi.BI_ERR_UNSUPPORTED
    assert L.bi_matmul(d, 8, d, 8, 0, d, 8, 0, 1 << 31, 8, 8, None) == bi.BI_ERR_UNSUPPORTED
    # empty problems are no-ops, even with null pointers
    assert L.bi_matmul(None, 0, None, 0, 0, None, 0, 0, 0, 8, 8, None) == bi.BI_OK
    assert L.bi_matmul(None, 0, None, 0, 0, None, 0, 0, 4, 0, 8, None) == bi.BI_OK


def test_rmsnorm_argument_errors_before_launch(L):
    d = ctypes.c_void_p(16)
    f = ctypes.c_float
    assert L.bi_rmsnorm(d, 8, d, d, 8, 0, -1, 8, f(1e-5), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(d, 8, d, d, 8, 0, 1, 0, f(1e-5), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(d, 8, d, d, 8, 0, 1, 8, f(-1.0), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(d, 8, d, d, 8, 0, 1, 8, f(float("nan")), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(d, 4, d, d, 8, 0, 1, 8, f(1e-5), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(None, 8, d, d, 8, 0, 1, 8, f(1e-5), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(d, 8, d, d, 8, 5, 1, 8, f(1e-5), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rmsnorm(None, 8, None, None, 8, 0, 0, 8, f(1e-5), None) == bi.BI_OK


def _verify(L, **kw):
    d = ctypes.c_void_p(256)
    a = dict(q=d, k=d, v=d, num_pages=4, bt=d, max_pages=4, sl=d, cu=d, batch=1, total_q=2,
             max_q=2, max_seq_len=200, hq=32, hkv=8, D=128, page=64, scale=0.1, out=d, lse=None,
             ws=d, ws_bytes=1 << 30)
    a.update(kw)
    return L.bi_verify_block(a["q"], a["k"], a["v"], a["num_pages"], a["bt"], a["max_pages"],
                             a["sl"], a["cu"], a["batch"], a["total_q"], a["max_q"],
                             a["max_seq_len"], a["hq"], a["hkv"], a["D"], a["page"],
                             ctypes.c_float(a["scale"]), a["out"], a["lse"], a["ws"],
                             a["ws_bytes"], None)


def test_attention_argument_errors_before_launch(L):
    assert _verify(L, D=96) == bi.BI_ERR_UNSUPPORTED
    assert _verify(L, page=32) == bi.BI_ERR_UNSUPPORTED
    assert _verify(L, hq=30) == bi.BI_ERR_INVALID_ARG
    assert _verify(L, max_q=9) == bi.BI_ERR_UNSUPPORTED
    assert _verify(L, max_q=8, total_q=8, hq=64, hkv=8) == bi.BI_ERR_UNSUPPORTED  # 8*8 rows
    assert _verify(L, max_seq_len=257 * 64, max_pages=256) == bi.BI_ERR_INVALID_ARG
    assert _verify(L, total_q=3) == bi.BI_ERR_INVALID_ARG
    assert _verify(L, cu=None) == bi.BI_ERR_INVALID_ARG
    assert _verify(L, ws_bytes=16) == bi.BI_ERR_INVALID_ARG
    assert "workspace" in _err(L)
    assert _verify(L, scale=float("inf")) == bi.BI_ERR_INVALID_ARG
    assert _verify(L, q=ctypes.c_void_p(258)) == bi.BI_ERR_UNSUPPORTED
    assert _verify(L, batch=0, total_q=0) == bi.BI_OK


def _prefill(L, **kw):
    d = ctypes.c_void_p(256)
    a = dict(q=d, k=d, v=d, num_pages=4, bt=d, max_pages=4, sl=d, cu=d, batch=1, total_q=200,
             max_q=200, max_seq_len=200, hq=32, hkv=8, D=128, page=64, scale=0.1, out=d,
             lse=None, ws=d, ws_bytes=1 << 30)
    a.update(kw)
    return L.bi_prefill_attn(a["q"], a["k"], a["v"], a["num_pages"], a["bt"], a["max_pages"],
                             a["sl"], a["cu"], a["batch"], a["total_q"], a["max_q"],
                             a["max_seq_len"], a["hq"], a["hkv"], a["D"], a["page"],
                             ctypes.c_float(a["scale"]), a["out"], a["lse"], a["ws"],
                             a["ws_bytes"], None)


def test_prefill_argument_errors_before_launch(L):
    """Blocks wider than a verify block are its purpose; a group size that does not divide
    the 128-row tile, max_q < 1 and the verify block's other rules are refused."""
    assert _prefill(L, hq=24, hkv=8) == bi.BI_ERR_UNSUPPORTED     # G = 3
    assert "divide 128" in _err(L)
    assert _prefill(L, max_q=0) == bi.BI_ERR_INVALID_ARG
    assert _prefill(L, D=96) == bi.BI_ERR_UNSUPPORTED
    assert _prefill(L, total_q=201) == bi.BI_ERR_INVALID_ARG       # > batch * max_q
    assert _prefill(L, cu=None) == bi.BI_ERR_INVALID_ARG
    assert _prefill(L, ws_bytes=16) == bi.BI_ERR_INVALID_ARG
    assert _prefill(L, q=ctypes.c_void_p(258)) == bi.BI_ERR_UNSUPPORTED
    assert _prefill(L, batch=0, total_q=0) == bi.BI_OK


def test_workspace_size_formula(L):
    # one (m, l, o[D]) fp32 partial per (token, head, 512-key chunk), then one 4-byte item
    # counter per (token, head), each part rounded up to 16 bytes
    r16 = lambda n: -(-n // 16) * 16  # noqa: E731
    assert L.bi_attn_workspace_size(8, 32, 128, 65540) == r16(8 * 32 * 129 * 130 * 4) + r16(8 * 32 * 4)
    assert L.bi_attn_workspace_size(1, 4, 64, 128) == r16(1 * 4 * 1 * 66 * 4) + r16(4 * 4)
    assert L.bi_attn_workspace_size(3, 1, 64, 64) == r16(3 * 66 * 4) + r16(3 * 4)
    assert L.bi_attn_workspace_size(1, 4, 96, 128) == 0
    assert L.bi_attn_workspace_size(1, 4, 64, 0) == 0


def test_selftest_rejects_bad_timeout(L):
    assert L.bi_selftest_wait_timeout(10, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_selftest_wait_timeout(10 ** 11, None) == bi.BI_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    """There is no CPU path: CPU tensors are refused, never computed on the host."""
    import torch
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        bi.matmul(x, torch.zeros(8, 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        bi.rmsnorm(x, torch.ones(8, dtype=torch.bfloat16), 1e-5)


def test_glue_argument_errors_before_launch(L):
    d = 1 << 20  # a fake, 16-byte aligned address: nothing may touch it
    f = ctypes.c_float
    # embedding: vocab < 1, hidden not a multiple of 8, ldo < hidden, null ids
    assert L.bi_embedding(d, 0, 64, d, 1, d, 64, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_embedding(d, 10, 60, d, 1, d, 64, None) == bi.BI_ERR_UNSUPPORTED
    assert L.bi_embedding(d, 10, 64, d, 1, d, 32, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_embedding(d, 10, 64, None, 1, d, 64, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_embedding(d + 8, 10, 64, d, 1, d, 64, None) == bi.BI_ERR_UNSUPPORTED
    assert L.bi_embedding(None, 10, 64, None, 0, None, 64, None) == bi.BI_OK  # n = 0
    # rope: head_dim not a multiple of 16, theta <= 0, no cu_q with total_q != batch
    assert L.bi_rope(d, 96, 1, 4, 24, d, None, 1, f(1e4), None) == bi.BI_ERR_UNSUPPORTED
    assert L.bi_rope(d, 128, 1, 2, 64, d, None, 1, f(0.0), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rope(d, 128, 2, 2, 64, d, None, 1, f(1e4), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rope(d, 64, 1, 2, 64, d, None, 1, f(1e4), None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_rope(d, 128, 1, 2, 64, d, None, 0, f(1e4), None) == bi.BI_ERR_INVALID_ARG
    # swiglu: stride < inter, inter not a multiple of 8
    assert L.bi_swiglu(d, 8, d, 16, d, 16, 1, 16, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_swiglu(d, 12, d, 12, d, 12, 1, 12, None) == bi.BI_ERR_UNSUPPORTED
    # add: n < 0, misaligned
    assert L.bi_add(d, d, d, -1, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_add(d + 2, d, d, 8, None) == bi.BI_ERR_UNSUPPORTED
    # argmax: n < 1, ld < n, ld not a multiple of 4
    assert L.bi_argmax(d, 8, 1, 0, d, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_argmax(d, 4, 1, 8, d, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_argmax(d + 2, 10, 1, 10, d, None) == bi.BI_ERR_INVALID_ARG
    assert "bi_argmax" in L.bi_last_error_message().decode()
    assert L.bi_argmax(d, 8, 0, 8, d, None) == bi.BI_OK  # rows = 0


def test_rowwise_argument_errors_before_launch(L):
    d = 1 << 20  # a fake, 16-byte aligned address: nothing may touch it
    assert L.bi_log_softmax(d, 8, d, 8, 1, 0, None) == bi.BI_ERR_INVALID_ARG       # n < 1
    assert L.bi_log_softmax(d, 4, d, 8, 1, 8, None) == bi.BI_ERR_INVALID_ARG       # ldx < n
    assert L.bi_log_softmax(d + 2, 8, d, 8, 1, 8, None) == bi.BI_ERR_INVALID_ARG   # misaligned
    assert L.bi_log_softmax(None, 8, d, 8, 1, 8, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_log_softmax(None, 8, None, 8, 0, 8, None) == bi.BI_OK              # rows = 0
    assert L.bi_mean(d, 8, 7, 1, 8, d, None) == bi.BI_ERR_INVALID_ARG              # dtype
    assert L.bi_mean(d, 4, bi.BI_F32, 1, 8, d, None) == bi.BI_ERR_INVALID_ARG      # ldx < n
    assert L.bi_mean(d + 1, 8, bi.BI_BF16, 1, 8, d, None) == bi.BI_ERR_INVALID_ARG
    assert L.bi_mean(d, 8, bi.BI_F32, 1, 8, None, None) == bi.BI_ERR_INVALID_ARG
    assert "bi_mean" in L.bi_last_error_message().decode()
