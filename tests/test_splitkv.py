"""Split-KV (keys split into ranges, results merged): GPU parity against the oracle.

The merged result must equal attention over all keys (the oracle's
definition), with the same gates as the unsplit path.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from test_parity import sample_rows
from workloads import WORKLOADS, make_inputs, make_qkv, rising_norm_order

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,dtype,sig,splits", [
    (1, 2, 1000, 128, "bf16", 3.0, 2),
    (1, 3, 777, 128, "f16", 1.0, 3),
    (2, 1, 2048, 64, "bf16", 1.0, 5),
    (1, 1, 300, 64, "f16", 2.0, 9),      # clamped to 3 ranges, the last one ragged
    (1, 2, 4096, 128, "bf16", 3.0, 0),   # automatic count
    (1, 2, 1000, 256, "bf16", 3.0, 2),   # d = 256: 128-row Q tiles, 64-key tiles
    (2, 1, 1111, 256, "f16", 1.0, 4),
    (1, 1, 300, 256, "bf16", 2.0, 9),    # 5 tiles of 64 keys: clamped to 5 ranges, the last one ragged
    (1, 3, 2048, 256, "bf16", 3.0, 0),   # automatic count (24 units on 152 SMs: split)
])
def test_splitkv_parity(B, H, N, d, dtype, sig, splits):
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=17, wid=11000 + N + splits)
    if sig > 1:
        k, v = rising_norm_order(k, v)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, dtype)
    assert res["ok"], res


def test_splitkv_long_sequence_workload_uniform_split_whole():
    """B=1 H=8 N=16384 with every unit split four ways (two launches: the
    partial pass and the merge), every output against the oracle."""
    from whole_parity import compare_whole, oracle_full
    w = WORKLOADS["b1h8n16384d128_bf16"]
    q, k, v = make_inputs(w)
    assert fa.fa_fwd_splitkv_launches(w.B, w.H, w.N, w.d, 4) == 2
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), num_splits=4)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref, _ = oracle_full(w, q, k, v)
    res = compare_whole(o, lse, o_ref, lse_ref, "bf16", label=f"{w.name} uniform 4-way split")
    assert res["ok"], res


def test_splitkv_workspace_errors():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 1000, 128, "bf16", seed=1, wid=11999))
    o, lse = torch.empty_like(q), torch.empty((1, 2, 1000), device="cuda")
    need = fa.fa_fwd_splitkv_workspace_size(1, 2, 1000, 128, 4)
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 2, 1000, 128, 0.088, fa.FA_BF16, 4)
    assert fa.fa_fwd_splitkv(*args, None, need, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 1, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr() + 16, need, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, None) == fa.FA_OK
    torch.cuda.synchronize()
    # a split count of 1 needs no workspace
    assert fa.fa_fwd_splitkv(*args[:-1], 1, None, 0, None) == fa.FA_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (1, 4, 10000, 128, "bf16"),   # 160 units: on 152 SMs one full wave, the 8 left over split 16 ways
    (1, 2, 20000, 128, "f16"),    # N not a multiple of 256: the last Q block of a head is partial
    (1, 4, 16384, 256, "bf16"),   # d = 256: 512 units of 128 rows, 3 full waves, the 56 left split 2 ways
])
def test_splitkv_tail_plan(B, H, N, d, dtype):
    """num_splits = 0 on shapes whose units end in a partial last wave: the
    full waves run unsplit, the last wave's units split and merged. Rows of
    the first and last heads (both sides of the split) against the oracle."""
    assert fa.fa_fwd_splitkv_num_splits(B, H, N, d) >= 2
    assert fa.fa_fwd_splitkv_launches(B, H, N, d, 0) == 3
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=1.5, seed=31, wid=11500 + N)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), num_splits=0)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rng = np.random.default_rng(N)
    heads = [(0, 0), (B - 1, H - 1)] + ([(B - 1, H - 2)] if H > 1 else [])
    rows = []
    for b, h in heads:
        for i in sorted({0, 255, 256, N - 1, N // 2, *rng.integers(0, N, 8).tolist()}):
            rows.append((b, h, i))
    o_ref, lse_ref = oracle.attn_rows(q, k, v, rows)
    oc, lc = o.cpu().double().numpy(), lse.cpu().double().numpy()
    res = compare(np.stack([oc[b, h, i] for b, h, i in rows]), np.array([lc[b, h, i] for b, h, i in rows]),
                  o_ref, lse_ref, dtype)
    assert res["ok"], res
    assert np.all(np.isfinite(oc)) and np.all(np.isfinite(lc))


def test_splitkv_tail_plan_workspace_covers_only_the_tail_rows():
    """Under the tail plan the partial buffers hold the split rows only: the
    workspace is smaller than the one every row split alike would need, a
    byte less is refused, and the launches write nothing past its end."""
    B, H, N, d = 1, 4, 10000, 128
    assert fa.fa_fwd_splitkv_launches(B, H, N, d, 0) == 3
    splits = fa.fa_fwd_splitkv_num_splits(B, H, N, d)
    need = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 0)
    assert 0 < need < fa.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=1.5, seed=32, wid=11600)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = torch.empty_like(qc), torch.empty((B, H, N), device="cuda")
    ws = torch.full((need + 65536,), 0x5A, dtype=torch.uint8, device="cuda")
    args = (qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, d ** -0.5,
            fa.FA_BF16, 0)
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 1, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, None) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert bool((ws[need:] == 0x5A).all())
    o_ref, lse_ref = fa.attention(qc, kc, vc, num_splits=1)
    torch.cuda.synchronize()
    # the same rows as the unsplit pass up to the merge's rounding
    assert float((o.float() - o_ref.float()).abs().max()) <= 1e-2
    assert float((lse - lse_ref).abs().max()) <= 1e-4 * max(1.0, float(lse_ref.abs().max()))


def test_splitkv_plan_matches_the_device_queries():
    """fa_fwd_splitkv_plan with this device's SM count agrees with the queries
    that read the device: split count, launches, workspace."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, H, N, d in [(1, 8, 16384, 128), (8, 32, 4096, 128), (8, 12, 2048, 128), (1, 4, 10240, 128),
                       (2, 2, 1000, 64), (4, 16, 4096, 256), (1, 1, 1280, 64)]:
        for ns in (0, 1, 3):
            rc, p = fa.fa_fwd_splitkv_plan(B, H, N, d, ns, sms)
            assert rc == fa.FA_OK
            assert p["launches"] == fa.fa_fwd_splitkv_launches(B, H, N, d, ns)
            assert p["workspace_bytes"] == fa.fa_fwd_splitkv_workspace_size(B, H, N, d, ns)
            if ns == 0:
                assert p["splits"] == fa.fa_fwd_splitkv_num_splits(B, H, N, d)


def _stream_plan_here(B, H, N):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, sp = fa.fa_fwd_stream_plan(B, H, N, 128, sms)
    assert rc == fa.FA_OK
    if sp["ctas"] == 0:
        pytest.skip(f"the plan does not stream this shape's tail on {sms} SMs")
    return sp


@pytest.mark.parametrize("B,H,N,dtype,sig", [
    (1, 20, 2048, "bf16", 3.0),   # 160 units: one full round, 8 units (128 tiles) over 76 CTAs, up to 10 pieces
    (3, 7, 2048, "f16", 1.0),     # 168 units: one full round, 16 units (256 tiles) over 76 CTAs
    (1, 2, 4096, "bf16", 2.0),    # 32 units: no full round, every unit streamed over 126 CTAs
])
def test_stream_tail_parity(B, H, N, dtype, sig):
    """The streamed tail of the automatic plan (persistent kernel: full rounds
    of whole units, then the left-over units' K/V tiles cut into one range
    per CTA, the cut units merged): every output against the oracle, and
    the rows of the whole units bit-identical to the unsplit pass, which
    computes them with the same code."""
    sp = _stream_plan_here(B, H, N)
    q, k, v = make_qkv(B, H, N, 128, dtype, sigma_qk=sig, seed=41, wid=12000 + N + H)
    if sig > 1:
        k, v = rising_norm_order(k, v)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.attention(qc, kc, vc, num_splits=0)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, dtype)
    assert res["ok"], res
    o1, lse1 = fa.attention(qc, kc, vc, num_splits=1)
    torch.cuda.synchronize()
    rows = sp["unit0"] * 256  # units are numbered head by head, 256 rows each
    assert torch.equal(o.view(-1, 128)[:rows], o1.view(-1, 128)[:rows])
    assert torch.equal(lse.view(-1)[:rows], lse1.view(-1)[:rows])


def test_stream_tail_workspace_bound():
    """The streamed path needs exactly the reported workspace: a byte less is
    refused, and nothing is written past its end."""
    B, H, N, d = 1, 20, 2048, 128
    _stream_plan_here(B, H, N)
    need = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 0)
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=1.0, seed=42, wid=12100)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = torch.empty_like(qc), torch.empty((B, H, N), device="cuda")
    ws = torch.full((need + 65536,), 0x5A, dtype=torch.uint8, device="cuda")
    args = (qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, d ** -0.5,
            fa.FA_BF16, 0)
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 1, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, None) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert bool((ws[need:] == 0x5A).all())
    o1, lse1 = fa.attention(qc, kc, vc, num_splits=1)
    torch.cuda.synchronize()
    assert float((o.float() - o1.float()).abs().max()) <= 1e-2
    assert float((lse - lse1).abs().max()) <= 1e-4 * max(1.0, float(lse1.abs().max()))


def test_stream_tail_noalloc_matches_workspace_call():
    """fa_fwd_splitkv_noalloc takes the streamed tail through the built-in
    scratch: bit-identical to the caller-workspace call, twice in a row."""
    B, H, N, d = 3, 7, 2048, 128
    _stream_plan_here(B, H, N)
    q, k, v = make_qkv(B, H, N, d, "f16", sigma_qk=1.0, seed=43, wid=12200)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = fa.attention(qc, kc, vc, num_splits=0)
    for _ in range(2):
        o, lse = torch.empty_like(qc), torch.empty((B, H, N), device="cuda")
        rc = fa.fa_fwd_splitkv_noalloc(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, H, N, d, d ** -0.5, fa.FA_F16, 0)
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
