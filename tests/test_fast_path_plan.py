"""Host logic of the batch-invariant limit's gate, without a GPU: which configuration a
call runs inside and outside the limit ("Fix/speculative shape invariance",
ml-explore/mlx PR 4279, section Changes: inside the limit the canonical reduction is
required; above it, or with the limit at 0, the optimized paths stay in use)."""
import pytest

import invariant_bi_matmul_gb300 as bi

ATTN = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


@pytest.fixture
def limit():
    old = bi.get_batch_invariant_limit()
    yield bi.set_batch_invariant_limit
    bi.set_batch_invariant_limit(old)


def ws(total_q, L, factor=1):
    return factor * bi.attn_workspace_size(total_q, 32, 128, L)


def chunk(B, q, L, w):
    return bi.attn_chunk(B, B * q, q, L, workspace_bytes=w, **ATTN)


def test_inside_the_limit_everything_is_the_invariant_configuration(limit):
    limit(1 << 20)
    for M, N, K in [(1, 4096, 4096), (8, 1024, 4096), (128, 4096, 14336), (4, 64, 4160)]:
        for lay in ("nk", "kn"):
            assert bi.matmul_splits(M, N, K, lay) == 1
    for B, q, L in [(1, 1, 1028), (1, 8, 65540), (8, 1, 65540), (64, 4, 8196)]:
        assert chunk(B, q, L, ws(B * q, L, 8)) == bi.ATTN_CHUNK


def test_limit_boundary_is_inclusive(limit):
    limit(8)
    assert bi.matmul_splits(8, 2048, 4096) == 1
    assert bi.matmul_splits(9, 2048, 4096) > 1
    assert chunk(1, 8, 1028, ws(8, 1028, 8)) == bi.ATTN_CHUNK
    limit(7)
    assert chunk(1, 8, 1028, ws(8, 1028, 8)) != bi.ATTN_CHUNK


def test_split_k_outside_the_limit(limit):
    limit(0)  # disabled: every call may take the fast path
    # one M-tile whose 32-column tiles leave most of the 152 SMs idle: split
    assert bi.matmul_splits(1, 2048, 4096) == 2          # 64 tiles
    assert bi.matmul_splits(128, 2048, 4096, "kn") == 2
    assert bi.matmul_splits(8, 1024, 4096) == 4          # 32 tiles
    assert bi.matmul_splits(8, 512, 4096) == 8           # 16 tiles, capped at 8 per tile
    # two M-tiles, or enough column tiles, or a single K-block: no split
    assert bi.matmul_splits(1, 4096, 4096) == 1          # 128 tiles
    assert bi.matmul_splits(129, 4096, 4096) == 1
    assert bi.matmul_splits(8, 14336, 4096) == 1
    assert bi.matmul_splits(8, 128256, 4096) == 1
    assert bi.matmul_splits(4, 64, 64) == 1
    # the reduction slots (rows x 32 fp32 per extra CTA) must leave the ring room
    assert 2 <= bi.matmul_splits(100, 1024, 4096) < 8
    # no CTA without K-blocks, whatever the split
    for K in (64 * 3, 64 * 9 + 5, 4160, 14336):
        s = bi.matmul_splits(2, 1024, K)
        assert 1 <= s <= min(8, -(-K // 64))


def test_attention_chunk_outside_the_limit(limit):
    limit(0)
    for B, q, L in [(1, 1, 1028), (1, 8, 65540), (8, 1, 65540), (32, 4, 8196), (64, 1, 16388)]:
        c = chunk(B, q, L, ws(B * q, L, 8))
        assert c in (64, 128, 256, 512, 1024, 2048)
        # with the invariant-size workspace no chunk shorter than the invariant one fits
        assert chunk(B, q, L, ws(B * q, L)) >= bi.ATTN_CHUNK
    # a short context at batch 1 leaves SMs idle with 512-key chunks: shorter ones win
    assert chunk(1, 1, 1028, ws(1, 1028, 8)) < bi.ATTN_CHUNK
    # many long sequences: longer chunks (fewer partials to write and merge)
    assert chunk(8, 1, 65540, ws(8, 65540)) > bi.ATTN_CHUNK
    # the choice follows the load: the same query length at another batch size can differ
    assert len({chunk(B, 1, 65540, ws(B, 65540, 8)) for B in (1, 8)}) == 2


def test_plan_rejects_invalid_sizes(limit):
    limit(0)
    assert bi.matmul_splits(0, 64, 64) == 0
    assert bi.matmul_splits(1, 64, 64, num_sms=0) == 0
    assert bi.attn_chunk(1, 2, 1, 100, 32, 8, 128, 1 << 20) == 0     # total_q > batch*max_q
    assert bi.attn_chunk(1, 1, 1, 100, 32, 8, 96, 1 << 20) == 0      # head_dim
    assert bi.attn_chunk(1, 1, 1, 100, 30, 8, 128, 1 << 20) == 0     # heads not a multiple
