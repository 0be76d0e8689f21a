"""Split-KV partial buffers: the row indexing of the split epilogue and of
the merge, restated from the kernels' index expressions and checked on the
CPU against the workspace the host plans (`fa_fwd_splitkv_plan`).

Work unit u covers Q block u % nqb of head u // nqb (q = 256 rows; 128 at
head dimension 256). Under a plan whose split units start at unit `first`,
their rows start at row0 = (first // nqb) * N + (first % nqb) * q, and the
epilogue of key
range s writes row r (< N) of head bh to partial row
s * (B*H*N - row0) + (bh * N + r - row0). The merge reads, for every output
row from row0 on, the same index for each s. The check: over every split
unit, every key range and every row, the partial rows written are exactly
[0, splits * (B*H*N - row0)), each once, inside the planned workspace, and
they are the rows the merge reads.
"""
import numpy as np
import pytest

import exact_attention_87_gb300 as fa
from exact_attention_87_gb300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fa.lib()


def _qblock(u, nqb, causal, num_splits, qunit_count):
    """The Q block of work unit u of a split launch, restated from the
    kernels: every split launch keeps the natural order. (Only a causal
    launch over every unit unsplit reorders its units, longest first within
    windows of heads; test_cta_order.py checks that order.)"""
    heavy_first = causal and num_splits == 1 and qunit_count == 0
    assert not heavy_first, "the split launches checked here keep the natural order"
    return u % nqb


def _qrows(d):
    """Q rows of one work unit: two 128-row sub-tiles, or one tile at d = 256."""
    return 128 if d == 256 else 256


def _written(B, H, N, first, splits, causal=False, d=128):
    q = _qrows(d)
    nqb = -(-N // q)
    units = B * H * nqb
    row0 = (first // nqb) * N + (first % nqb) * q
    span = B * H * N - row0
    idx = []
    for u in range(first, units):
        bh = u // nqb
        qb = _qblock(u, nqb, causal, splits, units - first)
        rows = np.arange(qb * q, min(qb * q + q, N))
        for s in range(splits):
            idx.append(s * span + (bh * N + rows - row0))
    return np.concatenate(idx) if idx else np.zeros(0, dtype=np.int64), row0, span


@pytest.mark.parametrize("B,H,N,d,num_sms", [
    (1, 8, 16384, 128, 152), (1, 8, 16384, 128, 148), (8, 12, 2048, 128, 152), (1, 4, 10240, 128, 152),
    (1, 8, 16000, 128, 152), (1, 4, 10000, 128, 152), (1, 2, 20000, 128, 152), (3, 5, 1000, 64, 7), (2, 3, 4097, 64, 13), (1, 1, 300, 64, 1),
    (4, 16, 4096, 256, 152), (1, 4, 16384, 256, 152), (2, 3, 1000, 256, 7), (1, 1, 300, 256, 1),
])
@pytest.mark.parametrize("num_splits", [0, 2, 5])
@pytest.mark.parametrize("causal", [False, True])
def test_partial_rows_tile_the_planned_workspace(L, B, H, N, d, num_sms, num_splits, causal):
    """Also under the causal mask (fa_fwd_splitkv_ex), whose plan is the
    unmasked one: the split launches keep the natural unit order, so the tail
    plan's units still hold exactly the rows from row0 on."""
    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, d, num_splits, num_sms)
    assert rc == fa.FA_OK
    rc, sp = fa.fa_fwd_stream_plan(B, H, N, d, num_sms)
    if num_splits == 0 and sp["ctas"] > 0:
        # the streamed tail (its slots are checked in test_stream_tail.py); masked
        # calls take the key-range plan, whose workspace the reported size covers
        assert p["launches"] == 2 and p["first_split_unit"] == sp["unit0"]
        return
    if p["splits"] == 1:
        assert p["workspace_bytes"] == 0
        return
    idx, row0, span = _written(B, H, N, p["first_split_unit"], p["splits"], causal, d)
    # every partial row exactly once, no gap, no overlap
    assert len(idx) == p["splits"] * span
    assert np.array_equal(np.sort(idx), np.arange(p["splits"] * span))
    # inside the planned workspace: fp32 O rows (256-byte aligned block) then fp32 LSE rows
    o_bytes = (p["splits"] * span * d * 4 + 255) // 256 * 256
    assert o_bytes + p["splits"] * span * 4 == p["workspace_bytes"]
    # the merge reads row r >= row0 of range s at s * span + (r - row0): the same set
    merge = np.concatenate([s * span + np.arange(span) for s in range(p["splits"])])
    assert np.array_equal(np.sort(merge), np.sort(idx))
    # and the merged rows are exactly the split units' rows
    q = _qrows(d)
    nqb = -(-N // q)
    first = p["first_split_unit"]
    assert row0 == (first // nqb) * N + (first % nqb) * q and span == B * H * N - row0


def test_heavy_first_order_would_break_the_tail_plan():
    """Planted mistake: the causal heavy-first order applied to the split
    tail launch too. Its units would then write rows before row0, outside
    the partial buffers (negative partial rows)."""
    B, H, N, num_sms = 1, 8, 16000, 152
    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, 128, 0, num_sms)
    assert rc == fa.FA_OK and 0 < p["first_split_unit"] and p["launches"] == 3
    nqb = -(-N // 256)
    first = p["first_split_unit"]
    row0 = (first // nqb) * N + (first % nqb) * 256
    bad = []
    for u in range(first, B * H * nqb):
        bh, qb = u // nqb, nqb - 1 - u % nqb   # reversed
        bad.append(bh * N + qb * 256 - row0)
    assert min(bad) < 0
