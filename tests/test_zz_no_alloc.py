"""bi_verify_block_static_ws: verify attention for callers that cannot allocate device
memory (work recorded into someone else's CUDA graph, allocator-free runtimes, real-time
paths).  It runs with the library's own fixed device workspace instead of one the caller
passes.  Checked here through the C ABI against bi_verify_block with a caller-provided
workspace, on two calls in a row (the fixed workspace keeps the previous call's contents,
which must not leak into the next result).

The file is named so that pytest collects it last; it also passes run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _block(seq_lens, q_lens, seed, dev):
    p = inputs.paged_inputs(seq_lens, q_lens, Hq=32, Hkv=8, D=128, seed=seed)
    t = {k: getattr(p, k).to(dev) for k in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                            "block_table", "seq_lens", "cu_q")}
    bi.kv_append(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["block_table"],
                 t["seq_lens"], t["cu_q"])
    return t, max(q_lens), max(seq_lens)


def _static_call(t, max_q, max_len, out, lse):
    """bi_verify_block_static_ws through the C ABI (no workspace argument)."""
    L = bi.lib()
    T, hq, d = t["q"].shape
    num_pages, hkv, page, _ = t["k_cache"].shape
    return L.bi_verify_block_static_ws(
        t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(), num_pages,
        t["block_table"].data_ptr(), t["block_table"].shape[1], t["seq_lens"].data_ptr(),
        t["cu_q"].data_ptr(), t["seq_lens"].shape[0], T, max_q, max_len, hq, hkv, d, page,
        ctypes.c_float(1.0 / np.sqrt(d)), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_static_workspace_matches_caller_workspace_twice(dev):
    cases = [_block([8196, 700, 1028], [8, 3, 4], seed=301, dev=dev),
             _block([65540], [8], seed=302, dev=dev)]
    for t, max_q, max_len in cases:
        ref, ref_lse = bi.verify_block(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                       t["seq_lens"], t["cu_q"], max_q=max_q,
                                       max_seq_len=max_len, scale=1.0 / np.sqrt(128))
        for _ in range(2):  # the second call sees the first call's leftovers in the scratch
            out = torch.full_like(ref, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            assert _static_call(t, max_q, max_len, out, lse) == bi.BI_OK
            torch.cuda.synchronize()
            check_bf16(out, ref.float().cpu().numpy(), "static workspace vs caller workspace")
            assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-6, atol=1e-6)
            # same kernels, same arithmetic: the bits agree as well
            assert bits_equal(out, ref) and bits_equal(lse, ref_lse)
    assert bi.device_status() == bi.BI_OK


def test_static_workspace_refuses_blocks_beyond_its_size(dev):
    """A valid block too large for the scratch: 64 sequences of 65,540 keys with verify
    blocks of 8 (512 tokens x 32 heads x 129 chunks of partials, far above 32 MiB).  The
    block tables all point at four shared pages, so the block costs no memory."""
    B, L, q = 64, 65540, 8
    need = bi.attn_workspace_size(B * q, 32, 128, L)
    assert need > bi.STATIC_WS_BYTES
    max_pages = -(-L // 64)
    kc = torch.zeros(4, 8, 64, 128, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    bt = (torch.arange(B * max_pages, dtype=torch.int32, device=dev) % 4).view(B, max_pages)
    sl = torch.full((B,), L, dtype=torch.int32, device=dev)
    cu = torch.arange(0, B * q + 1, q, dtype=torch.int32, device=dev)
    qt = torch.zeros(B * q, 32, 128, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(qt)
    lse = torch.empty(B * q, 32, dtype=torch.float32, device=dev)
    L_ = bi.lib()
    rc = L_.bi_verify_block_static_ws(
        qt.data_ptr(), kc.data_ptr(), vc.data_ptr(), 4, bt.data_ptr(), max_pages, sl.data_ptr(),
        cu.data_ptr(), B, B * q, q, L, 32, 8, 128, 64, ctypes.c_float(0.1), out.data_ptr(),
        lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == bi.BI_ERR_UNSUPPORTED
    assert "static scratch" in L_.bi_last_error_message().decode()
    assert bi.device_status() == bi.BI_OK


def test_static_workspace_outside_the_limit_matches_exact_workspace(dev):
    """With the limit at 0 the chunk length follows the workspace size: the entry point
    gives the bits of bi_verify_block handed exactly bi_attn_workspace_size() bytes."""
    t, max_q, max_len = _block([8196, 16388], [8, 8], seed=304, dev=dev)
    old = bi.get_batch_invariant_limit()
    bi.set_batch_invariant_limit(0)
    try:
        T = t["q"].shape[0]
        need = bi.attn_workspace_size(T, 32, 128, max_len)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        ref, ref_lse = bi.verify_block(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                       t["seq_lens"], t["cu_q"], max_q=max_q,
                                       max_seq_len=max_len, scale=1.0 / np.sqrt(128),
                                       workspace=ws)
        out = torch.empty_like(ref)
        lse = torch.empty_like(ref_lse)
        assert _static_call(t, max_q, max_len, out, lse) == bi.BI_OK
        torch.cuda.synchronize()
    finally:
        bi.set_batch_invariant_limit(old)
    assert bits_equal(out, ref) and bits_equal(lse, ref_lse)
