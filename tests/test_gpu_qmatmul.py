"""bi_qmatmul on the GPU: quantized W (mxfp4, nvfp4, mxfp8, affine 4/8-bit at group
sizes 32/64/128) against the oracle, including nvfp4 with K = 16 mod 32 ("Fix fp
quantized matmul corruption when the quantized dim is not a multiple of 32", Problem and
Fix) and ragged N; bit-identical to bi_matmul on the dequantized weights; rows bitwise
across M ("Fix/speculative shape invariance", the tester's comment: quantized matmul is
where the paths diverged most)."""
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


def _weights(fmt, N, K, gs, seed):
    q = inputs.Q_NAMES[fmt]
    wq, sc, b = inputs.quant_weights(q, N, K, gs, seed)
    affine = b is not None
    sc_np = inputs.bf16_bits(sc) if affine else sc.numpy()
    b_np = inputs.bf16_bits(b) if affine else None
    wd = oracle.dequantize(wq.numpy(), sc_np, b_np, q, gs, N, K)  # bf16 bits [N, K]
    return wq, sc, b, wd


def _run(dev, x, wq, sc, b, fmt, gs, K, out_dtype=None):
    return bi.qmatmul(x.to(dev), wq.to(dev), sc.to(dev), fmt, gs, K,
                      biases=None if b is None else b.to(dev), out_dtype=out_dtype)


@pytest.mark.parametrize("fmt,gs", FORMATS)
@pytest.mark.parametrize("M,N,K", [(8, 1024, 4096), (3, 200, 1040), (130, 96, 256)])
def test_qmatmul_matches_oracle(dev, fmt, gs, M, N, K):
    if K % gs:
        pytest.skip("K must be a multiple of the group size")
    x = inputs.normal_bf16((M, K), seed=M + K)
    wq, sc, b, wd = _weights(fmt, N, K, gs, seed=N + gs)
    ref = oracle.matmul(inputs.bf16_bits(x), wd, oracle.W_NK)
    wv = (wd.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.abs(x.float().numpy().astype(np.float64)) @ np.abs(wv).T
    y = _run(dev, x, wq, sc, b, fmt, gs, K)
    check_bf16(y, ref, f"qmatmul {fmt} gs{gs} {M}x{N}x{K}")
    y32 = _run(dev, x, wq, sc, b, fmt, gs, K, out_dtype=torch.float32)
    check_f32(y32, ref, scale, f"qmatmul fp32 {fmt} gs{gs} {M}x{N}x{K}")
    # the same instruction sequence as the dense GEMM on the dequantized weights
    wdt = torch.from_numpy(wd.view(np.int16)).view(torch.bfloat16).to(dev)
    assert bits_equal(y32, bi.matmul(x.to(dev), wdt, "nk", out_dtype=torch.float32))


@pytest.mark.parametrize("fmt,gs", [("mxfp4", 32), ("nvfp4", 16), ("affine4", 64)])
def test_qmatmul_rows_invariant_across_M(dev, fmt, gs):
    N, K = 4096, 4096
    x = inputs.normal_bf16((300, K), seed=77)
    wq, sc, b, _ = _weights(fmt, N, K, gs, seed=78)
    xd = x.to(dev)
    args = (wq.to(dev), sc.to(dev), fmt, gs, K)
    kw = {} if b is None else {"biases": b.to(dev)}
    full = bi.qmatmul(xd, *args, **kw)
    for M in (1, 2, 4, 8, 9, 64, 128, 129, 299):
        assert bits_equal(bi.qmatmul(xd[:M].contiguous(), *args, **kw), full[:M]), M
    old = bi.get_batch_invariant_limit()
    bi.set_batch_invariant_limit(0)  # one configuration: the limit changes nothing
    try:
        assert bits_equal(bi.qmatmul(xd[:8].contiguous(), *args, **kw), full[:8])
    finally:
        bi.set_batch_invariant_limit(old)


@pytest.mark.parametrize("fmt,gs", [("mxfp4", 32), ("affine8", 64)])
@pytest.mark.parametrize("M,N", [(1024, 4864), (1280, 4096)])
def test_qmatmul_wide_tiles_sampled(dev, fmt, gs, M, N):
    """Four 64-wide instruction tiles per CTA (three ring stages), one and two tiles per
    CTA: sampled rows against the oracle, and bit-identical to the dense GEMM."""
    K = 256
    x = inputs.normal_bf16((M, K), seed=M)
    wq, sc, b, wd = _weights(fmt, N, K, gs, seed=N)
    y = _run(dev, x, wq, sc, b, fmt, gs, K, out_dtype=torch.float32)
    assert bi.device_status() == bi.BI_OK
    rows = [0, 127, 128, M // 2, M - 1]
    ref = oracle.matmul(inputs.bf16_bits(x[rows]), wd, oracle.W_NK)
    wv = (wd.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.abs(x[rows].float().numpy().astype(np.float64)) @ np.abs(wv).T
    check_f32(y.cpu()[rows], ref, scale, f"wide qmatmul {fmt} {M}x{N}")
    wdt = torch.from_numpy(wd.view(np.int16)).view(torch.bfloat16).to(dev)
    assert bits_equal(y, bi.matmul(x.to(dev), wdt, "nk", out_dtype=torch.float32))


def test_qmatmul_repeat_and_guard_bands(dev):
    """Run-to-run identical, and nothing written outside y (the out-of-bounds store race of
    the tail tile is run-to-run nondeterminism)."""
    M, N, K = 5, 200, 1040
    x = inputs.normal_bf16((M, K), seed=90)
    wq, sc, _, _ = _weights("nvfp4", N, K, 16, seed=91)
    buf = torch.full((M + 2, N + 8), 7.0, dtype=torch.bfloat16, device=dev)
    out = buf[1:M + 1, :N]
    seen = set()
    for _ in range(30):
        bi.qmatmul(x.to(dev), wq.to(dev), sc.to(dev), "nvfp4", 16, K, out=out)
        seen.add(bytes(out.contiguous().view(torch.int16).cpu().numpy()))
    assert len(seen) == 1
    assert torch.all(buf[0] == 7.0) and torch.all(buf[M + 1] == 7.0)
    assert torch.all(buf[1:M + 1, N:] == 7.0)


def _same_or_both_nan(a, b):
    """Bitwise equality of two fp32 tensors, any NaN matching any NaN."""
    a, b = a.contiguous().cpu(), b.contiguous().cpu()
    same = a.view(torch.int32) == b.view(torch.int32)
    return bool(torch.all(same | (torch.isnan(a) & torch.isnan(b))))


def _block_enumeration(fmt, gs, K):
    """Every (scale code, element code) pair of a block format, one pair per W row: the
    row's only nonzero code sits at column (37 n) mod K, its group takes the scale code
    under test and the other groups the code of 1.0."""
    eight = fmt == "mxfp8"
    ncode = 256 if eight else 16
    N = 256 * ncode
    n = np.arange(N)
    kpos = (n * 37) % K
    codes = np.zeros((N, K), np.uint8)
    codes[n, kpos] = (n % ncode).astype(np.uint8)
    scales = np.full((N, K // gs), 0x38 if fmt == "nvfp4" else 127, np.uint8)
    scales[n, kpos // gs] = (n // ncode).astype(np.uint8)
    wq = codes if eight else (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return wq, scales, None, N


def _affine_enumeration(fmt, gs, K, seed):
    """Affine codes drawn uniformly with bf16 scales and biases of random sign, mantissa
    and exponent field 0 .. 0xE0 (subnormals included; no overflow)."""
    rng = np.random.default_rng(seed)
    N = 2048
    nb = K if fmt == "affine8" else K // 2
    wq = rng.integers(0, 256, (N, nb), dtype=np.uint8)

    def bf16_bits(shape):
        return ((rng.integers(0, 2, shape) << 15) | (rng.integers(0, 0xE1, shape) << 7)
                | rng.integers(0, 128, shape)).astype(np.uint16)
    return wq, bf16_bits((N, K // gs)), bf16_bits((N, K // gs)), N


def _padded(a, row_bytes=16):
    """The same values in rows padded to a multiple of row_bytes bytes (scales whose rows
    start on 16-byte boundaries travel with the codes by TMA; others are loaded by the
    converters)."""
    per = row_bytes // a.itemsize
    out = np.zeros((a.shape[0], -(-a.shape[1] // per) * per), a.dtype)
    out[:, :a.shape[1]] = a
    return out


@pytest.mark.parametrize("pad", [False, True])
@pytest.mark.parametrize("fmt,gs,K", [("mxfp4", 32, 64), ("nvfp4", 16, 64), ("mxfp8", 32, 64),
                                      ("affine4", 32, 64), ("affine4", 128, 128),
                                      ("affine8", 64, 64)])
def test_qmatmul_dequantizes_every_code_exactly(dev, fmt, gs, K, pad):
    """Identity X reads the dequantized W back out of Y (each Y element is one product
    W x 1 plus products with 0): every E2M1 / E4M3 code under every E8M0 / E4M3 scale
    code (NaN scales, overflow to infinity and subnormal results included) and affine
    codes under scales and biases of every exponent.  Y equals bi_matmul on the oracle's
    dequantized W bit for bit everywhere, and equals the oracle's values wherever the
    row holds no infinity or NaN and the value is zero or normal (whether the tensor
    cores keep subnormal inputs is theirs to decide, the same on both paths)."""
    q = inputs.Q_NAMES[fmt]
    if fmt.startswith("affine"):
        wq, sc, b, N = _affine_enumeration(fmt, gs, K, seed=K + gs)
    else:
        wq, sc, b, N = _block_enumeration(fmt, gs, K)
    wd = oracle.dequantize(wq, sc, b, q, gs, N, K)  # bf16 bits [N, K]
    x = torch.eye(K, dtype=torch.bfloat16, device=dev)
    to_dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)
    ng = K // gs
    sct = to_dev(_padded(sc) if pad else sc)[:, :ng]
    if b is not None:
        sct = sct.view(torch.bfloat16)
    bt = None if b is None else to_dev(_padded(b) if pad else b)[:, :ng].view(torch.bfloat16)
    yq = bi.qmatmul(x, to_dev(wq), sct, fmt, gs, K, biases=bt, out_dtype=torch.float32)
    wdt = torch.from_numpy(wd.view(np.int16)).view(torch.bfloat16).to(dev)
    yd = bi.matmul(x, wdt, "nk", out_dtype=torch.float32)
    assert _same_or_both_nan(yq, yd), f"{fmt}: quantized and dense paths differ"
    wv = (wd.astype(np.uint32) << 16).view(np.float32)         # [N, K]
    y = yd.cpu().numpy()                                       # [K, N]
    row_finite = np.all(np.isfinite(wv), axis=1)
    plain = (np.abs(wv) >= np.float32(2.0 ** -126)) | (wv == 0)
    mask = row_finite[None, :] & plain.T
    assert np.array_equal(y[mask], wv.T[mask]), f"{fmt}: values differ from the oracle"
    assert np.all(np.isnan(y[np.isnan(wv).T])), f"{fmt}: NaN weights lost"
    lone_inf = np.isinf(wv).T & (np.sum(~np.isfinite(wv), axis=1) == 1)[None, :]
    assert np.array_equal(y[lone_inf], wv.T[lone_inf]), f"{fmt}: infinite weights differ"
    if not fmt.startswith("affine"):  # the enumeration reached every kind of value
        assert mask.sum() > 0 and np.isnan(wv).sum() > 0
        assert (lone_inf.sum() > 0) == (fmt != "nvfp4")  # 6 x 448 stays finite


@pytest.mark.parametrize("fmt,gs", FORMATS)
@pytest.mark.parametrize("M,N,K", [(1, 300, 1600), (5, 200, 4160), (8, 96, 512)])
def test_qmatmul_small_m_multi_kblock_stages(dev, fmt, gs, M, N, K):
    """Small M with TMA-staged scales (rows padded to a 16-byte pitch): the kernel takes
    several K-blocks per stage, the last stage short (K = 1600: 25 K-blocks in stages of
    4; K = 4160: 65 in stages of 8).  Oracle parity, and the bits of the dense GEMM on the
    dequantized weights."""
    if K % gs:
        pytest.skip("K must be a multiple of the group size")
    wq, sc, b, wd = _weights(fmt, N, K, gs, seed=M + N + K)
    affine = b is not None
    sc_np = inputs.bf16_bits(sc) if affine else sc.numpy()
    sct = torch.from_numpy(_padded(sc_np).view(np.int16) if affine else _padded(sc_np))
    sct = sct.to(dev)[:, :K // gs]
    if affine:
        sct = sct.view(torch.bfloat16)
    bt = None
    if affine:
        bt = torch.from_numpy(_padded(inputs.bf16_bits(b)).view(np.int16)).to(dev)[:, :K // gs]
        bt = bt.view(torch.bfloat16)
    x = inputs.normal_bf16((M, K), seed=K + M)
    y32 = bi.qmatmul(x.to(dev), wq.to(dev), sct, fmt, gs, K, biases=bt, out_dtype=torch.float32)
    ref = oracle.matmul(inputs.bf16_bits(x), wd, oracle.W_NK)
    wv = (wd.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.abs(x.float().numpy().astype(np.float64)) @ np.abs(wv).T
    check_f32(y32, ref, scale, f"qmatmul staged {fmt} gs{gs} {M}x{N}x{K}")
    wdt = torch.from_numpy(wd.view(np.int16)).view(torch.bfloat16).to(dev)
    assert bits_equal(y32, bi.matmul(x.to(dev), wdt, "nk", out_dtype=torch.float32))
