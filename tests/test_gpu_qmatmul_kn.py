"""bi_qmatmul_ex in the natural layout (W stored [K, N], quantized along N: the qmm_n
orientation of "Fix fp quantized matmul corruption when the quantized dim is not a
multiple of 32", Problem and The three defects; both B orientations, "Fix/speculative
shape invariance", review thread).

Checked against the oracle (the same dequantization, rows along K instead of N), bit for
bit against the dense layout-KN GEMM on the dequantized weights, rows bitwise across M,
the nvfp4 tail (N = 16 mod 32) with guard bands and repeats, and every element code of
the block formats through an identity X."""
import numpy as np
import pytest
import torch

import oracle
from invariant_bi_matmul_gb300 import inputs
from tolerance import bits_equal, check_bf16, check_f32

pytestmark = pytest.mark.gpu

bi = pytest.importorskip("invariant_bi_matmul_gb300")

FORMATS = [("mxfp4", 32), ("nvfp4", 16), ("mxfp8", 32), ("affine4", 32), ("affine4", 64),
           ("affine4", 128), ("affine8", 32), ("affine8", 128)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _weights_kn(fmt, K, N, gs, seed):
    """Codes [K, row bytes] quantized along N, scales [K, N/gs] (and biases), and the
    oracle's dequantized W [K, N] (bf16 bits)."""
    q = inputs.Q_NAMES[fmt]
    wq, sc, b = inputs.quant_weights(q, K, N, gs, seed)  # rows = K, quantized dim = N
    affine = b is not None
    sc_np = inputs.bf16_bits(sc) if affine else sc.numpy()
    b_np = inputs.bf16_bits(b) if affine else None
    wd = oracle.dequantize(wq.numpy(), sc_np, b_np, q, gs, K, N)  # bf16 bits [K, N]
    return wq, sc, b, wd


def _run(dev, x, wq, sc, b, fmt, gs, K, N, out_dtype=None, out=None):
    return bi.qmatmul(x.to(dev), wq.to(dev), sc.to(dev), fmt, gs, K,
                      biases=None if b is None else b.to(dev), out_dtype=out_dtype, out=out,
                      layout="kn", N=N)


def _dense(wd, dev):
    return torch.from_numpy(wd.view(np.int16)).view(torch.bfloat16).to(dev)


@pytest.mark.parametrize("fmt,gs", FORMATS)
@pytest.mark.parametrize("M,N,K", [(8, 1024, 4096), (3, 256, 1040), (130, 128, 256),
                                   (1, 4096, 320)])
def test_qmatmul_kn_matches_oracle_and_dense_kn(dev, fmt, gs, M, N, K):
    if N % gs:
        pytest.skip("N must be a multiple of the group size")
    x = inputs.normal_bf16((M, K), seed=M + K)
    wq, sc, b, wd = _weights_kn(fmt, K, N, gs, seed=N + gs)
    ref = oracle.matmul(inputs.bf16_bits(x), wd, oracle.W_KN)
    wv = (wd.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.abs(x.float().numpy().astype(np.float64)) @ np.abs(wv)
    y = _run(dev, x, wq, sc, b, fmt, gs, K, N)
    check_bf16(y, ref, f"qmatmul kn {fmt} gs{gs} {M}x{N}x{K}")
    y32 = _run(dev, x, wq, sc, b, fmt, gs, K, N, out_dtype=torch.float32)
    check_f32(y32, ref, scale, f"qmatmul kn fp32 {fmt} gs{gs} {M}x{N}x{K}")
    # the dense layout-KN GEMM on the dequantized weights: the same bits
    assert bits_equal(y32, bi.matmul(x.to(dev), _dense(wd, dev), "kn", out_dtype=torch.float32))
    assert bi.device_status() == bi.BI_OK


@pytest.mark.parametrize("fmt,gs", [("mxfp4", 32), ("nvfp4", 16), ("affine8", 64)])
def test_qmatmul_kn_rows_invariant_across_M(dev, fmt, gs):
    N, K = 4096, 4096
    x = inputs.normal_bf16((300, K), seed=77).to(dev)
    wq, sc, b, _ = _weights_kn(fmt, K, N, gs, seed=78)
    kw = dict(biases=None if b is None else b.to(dev), layout="kn", N=N)
    args = (wq.to(dev), sc.to(dev), fmt, gs, K)
    full = bi.qmatmul(x, *args, out_dtype=torch.float32, **kw)
    for M in (1, 2, 8, 9, 64, 65, 128, 129, 299):
        part = bi.qmatmul(x[:M].contiguous(), *args, out_dtype=torch.float32, **kw)
        assert bits_equal(part, full[:M]), f"rows differ at M={M}"
    for i in (5, 128, 250):
        alone = bi.qmatmul(x[i:i + 1].contiguous(), *args, out_dtype=torch.float32, **kw)
        assert bits_equal(alone, full[i:i + 1]), f"row {i} differs alone"


def test_qmatmul_kn_nvfp4_tail_guard_bands_and_repeats(dev):
    """nvfp4 with N = 16 mod 32 (the tail the page's natural-layout kernel stored out of
    bounds) and ragged K: nothing written outside y, and one result over 30 repeats."""
    M, N, K = 5, 208, 1040
    x = inputs.normal_bf16((M, K), seed=90)
    wq, sc, _, wd = _weights_kn("nvfp4", K, N, 16, seed=91)
    buf = torch.full((M + 2, N + 16), 7.0, dtype=torch.bfloat16, device=dev)
    out = buf[1:M + 1, :N]
    seen = set()
    for _ in range(30):
        _run(dev, x, wq, sc, None, "nvfp4", 16, K, N, out=out)
        seen.add(bytes(out.contiguous().view(torch.int16).cpu().numpy()))
    assert len(seen) == 1
    assert torch.all(buf[0] == 7.0) and torch.all(buf[M + 1] == 7.0)
    assert torch.all(buf[1:M + 1, N:] == 7.0)
    ref = oracle.matmul(inputs.bf16_bits(x), wd, oracle.W_KN)
    check_bf16(out, ref, "nvfp4 tail")


def _same_or_both_nan(a, b):
    a, b = a.contiguous().cpu(), b.contiguous().cpu()
    same = a.view(torch.int32) == b.view(torch.int32)
    return bool(torch.all(same | (torch.isnan(a) & torch.isnan(b))))


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "mxfp8"])
def test_qmatmul_kn_every_element_code_through_identity(dev, fmt):
    """X = I: Y is W dequantized.  Every element code meets every scale code in the
    column it shares with no infinity or NaN (E8M0 scales 2^-20 .. 2^20, E4M3 scales of
    finite value), so Y equals the oracle's dequantized W exactly where the value is zero
    or normal; and Y equals the dense layout-KN GEMM on the oracle's W bit for bit."""
    q = inputs.Q_NAMES[fmt]
    eight = fmt == "mxfp8"
    gs = 16 if fmt == "nvfp4" else 32
    ncode = 256 if eight else 16
    K = 64
    N = ncode * gs  # column group g carries element code g in every row
    codes = np.zeros((K, N), np.uint8)
    n = np.arange(N)
    codes[:, :] = (n // gs) % ncode
    if eight:
        codes[(codes & 0x7F) == 0x7F] = 0  # no NaN element codes here
        wq = codes
    else:
        wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    rng = np.random.default_rng(5)
    if fmt == "nvfp4":
        sc = rng.integers(0x01, 0x7E, (K, N // gs)).astype(np.uint8)  # finite E4M3
    else:
        sc = rng.integers(127 - 20, 127 + 21, (K, N // gs)).astype(np.uint8)
    wd = oracle.dequantize(wq, sc, None, q, gs, K, N)
    x = torch.eye(K, dtype=torch.bfloat16, device=dev)
    y = bi.qmatmul(x, torch.from_numpy(wq).to(dev), torch.from_numpy(sc).to(dev), fmt, gs, K,
                   out_dtype=torch.float32, layout="kn", N=N)
    yd = bi.matmul(x, _dense(wd, dev), "kn", out_dtype=torch.float32)
    assert _same_or_both_nan(y, yd)
    wv = (wd.astype(np.uint32) << 16).view(np.float32)
    plain = (np.abs(wv) >= np.float32(2.0 ** -126)) | (wv == 0)
    col_ok = np.all(np.isfinite(wv), axis=0)[None, :]
    mask = plain & col_ok
    assert mask.mean() > 0.5
    assert np.array_equal(y.cpu().numpy()[mask], wv[mask])


def test_qmatmul_kn_rejects_bad_layouts(dev):
    x = torch.zeros(2, 64, dtype=torch.bfloat16, device=dev)
    wq = torch.zeros(64, 16, dtype=torch.uint8, device=dev)
    sc = torch.zeros(64, 1, dtype=torch.uint8, device=dev)
    with pytest.raises(bi.BIError) as e:  # N = 24 is not a multiple of the group size
        bi.qmatmul(x, wq, sc, "mxfp4", 32, 64, layout="kn", N=24)
    assert e.value.status == bi.BI_ERR_INVALID_ARG
    with pytest.raises(bi.BIError) as e:  # the rows of 16 bytes hold only 32 codes
        bi.qmatmul(x, wq, torch.zeros(64, 2, dtype=torch.uint8, device=dev), "mxfp4", 32, 64,
                   layout="kn", N=64)
    assert e.value.status == bi.BI_ERR_INVALID_ARG
