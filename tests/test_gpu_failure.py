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
