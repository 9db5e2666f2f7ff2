"""Failure detection without faulting the GPU: a kernel waits on an mbarrier nothing
arrives at, its bounded wait runs out, it latches BI_ERR_TIMEOUT in the device error
word and returns; the host reads the status and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def test_bounded_wait_times_out_and_context_survives(dev):
    assert bi.device_status() == bi.BI_OK
    bi.selftest_wait_timeout(50_000_000)             # 50 ms
    assert bi.device_status() == bi.BI_ERR_TIMEOUT
    assert bi.device_status() == bi.BI_OK            # reading clears the word
    x = torch.ones(2, 64, dtype=torch.bfloat16, device=dev)
    w = torch.ones(32, 64, dtype=torch.bfloat16, device=dev)
    y = bi.matmul(x, w, "nk", out_dtype=torch.float32)
    assert torch.all(y == 64.0)
    assert bi.device_status() == bi.BI_OK


# --------------------------------------------------------------------------------------
# The real kernels' bounded waits (book chapter "Batch-invariant kernels...": nothing
# here; this is the library's own failure detection).  A test-only budget shorter than a
# call's runtime makes the GEMM, attention and prefill kernels' waits run out; each must
# report BI_ERR_TIMEOUT through the error word, drain what it issued, free its tensor
# memory and return, and the next call with the default budget must give the same bits
# as before.

import math  # noqa: E402

import numpy as np  # noqa: E402

from invariant_bi_matmul_gb300 import inputs  # noqa: E402
from tolerance import bits_equal  # noqa: E402

SHORT_NS = 1000  # 1 us: far shorter than any of the calls below


@pytest.fixture
def default_budget_after():
    yield
    bi.selftest_set_wait_budget(0)
    bi.device_status()


def _times_out_then_recovers(call):
    ref = call()
    assert bi.device_status() == bi.BI_OK
    bi.selftest_set_wait_budget(SHORT_NS)
    call()
    status = bi.device_status()
    bi.selftest_set_wait_budget(0)
    assert status == bi.BI_ERR_TIMEOUT
    again = call()
    assert bi.device_status() == bi.BI_OK
    return ref, again


def test_selftest_budget_is_validated(dev):
    with pytest.raises(bi.BIError) as e:
        bi.selftest_set_wait_budget(10)
    assert e.value.status == bi.BI_ERR_INVALID_ARG
    bi.selftest_set_wait_budget(0)


def test_gemm_waits_run_out_and_the_next_call_matches(dev, default_budget_after):
    gi = inputs.gemm_inputs(2048, 4096, 4096, seed=2)
    x, w = gi.x.to(dev), gi.w_nk.to(dev)
    ref, again = _times_out_then_recovers(lambda: bi.matmul(x, w, "nk").clone())
    assert bits_equal(ref, again)


def test_quantized_gemm_waits_run_out_and_the_next_call_matches(dev, default_budget_after):
    N, K = 4096, 4096
    x = inputs.normal_bf16((2048, K), seed=3).to(dev)
    wq, sc, _ = inputs.quant_weights(inputs.Q_MXFP4, N, K, 32, seed=4)
    wq, sc = wq.to(dev), sc.to(dev)
    ref, again = _times_out_then_recovers(
        lambda: bi.qmatmul(x, wq, sc, "mxfp4", 32, K).clone())
    assert bits_equal(ref, again)


def test_verify_attention_waits_run_out_and_the_next_call_matches(dev, default_budget_after):
    L, q = 65540, 8
    p = inputs.paged_inputs([L], [q], Hq=32, Hkv=8, D=128, seed=5, device=dev)
    d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                             "seq_lens", "cu_q")}

    def call():
        o, l = bi.verify_block(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], d["cu_q"], max_q=q, max_seq_len=L,
                               scale=1.0 / math.sqrt(128))
        return torch.cat([o.float().reshape(-1), l.reshape(-1)])
    ref, again = _times_out_then_recovers(call)
    assert bits_equal(ref, again)


def test_prefill_waits_run_out_and_the_next_call_matches(dev, default_budget_after):
    L = 2048
    p = inputs.paged_inputs([L], [L], Hq=32, Hkv=8, D=128, seed=6, device=dev)
    d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                             "seq_lens", "cu_q")}

    def call():
        o, l = bi.prefill_attn(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], d["cu_q"], max_q=L, max_seq_len=L,
                               scale=1.0 / math.sqrt(128))
        return torch.cat([o.float().reshape(-1), l.reshape(-1)])
    ref, again = _times_out_then_recovers(call)
    assert bits_equal(ref, again)
    assert np.isfinite(ref.cpu().numpy()).all()
