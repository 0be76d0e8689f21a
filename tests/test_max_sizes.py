"""Large shapes: the longest single head, the widest grid, and a long backward.

These reach index ranges the benchmark workloads do not: 2^18 rows in one
head (row and tile indices, TMA coordinates, split-KV plans over 2048 tiles),
4096 heads of short sequences (a grid of 4096 units, head offsets up to
2^28 elements), a 65536-token head at d = 256, and a 16384-token head through
the backward pass. Each output is checked on sampled rows against the
oracle, which computes every sampled row from the whole head's keys.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from test_backward import gate
from workloads import make_dout, make_qkv

pytestmark = pytest.mark.gpu


def _rows(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = {(int(rng.integers(B)), int(rng.integers(H)), i) for i in edge if 0 <= i < N}
    rows |= {(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(n)}
    return sorted(rows)


def _check_rows(o, lse, q, k, v, rows, dtype):
    o_ref, lse_ref = oracle.attn_rows(q, k, v, rows)
    oc, lc = o.cpu().double().numpy(), lse.cpu().double().numpy()
    res = compare(np.stack([oc[b, h, i] for b, h, i in rows]), np.array([lc[b, h, i] for b, h, i in rows]),
                  o_ref, lse_ref, dtype)
    assert res["ok"], res
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


@pytest.mark.parametrize("num_splits", [1, 0])
def test_longest_single_head(num_splits):
    """B=1, H=1, N=262144, d=128, bf16: 2048 key tiles per Q block; unsplit and
    with the automatic split-KV plan."""
    B, H, N, d = 1, 1, 262144, 128
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=1.5, seed=41, wid=14600)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    _check_rows(o, lse, q, k, v, _rows(B, H, N, 12, seed=41), "bf16")


def test_widest_grid():
    """B=32, H=128, N=1024, d=64, fp16: 4096 heads, 4096 work units."""
    B, H, N, d = 32, 128, 1024, 64
    q, k, v = make_qkv(B, H, N, d, "f16", sigma_qk=2.0, seed=42, wid=14700)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rows = _rows(B, H, N, 40, seed=42) + [(B - 1, H - 1, N - 1), (B - 1, H - 1, 0)]
    _check_rows(o, lse, q, k, v, sorted(set(rows)), "f16")


def test_long_head_d256():
    """B=1, H=2, N=65536, d=256, bf16."""
    B, H, N, d = 1, 2, 65536, 256
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=1.5, seed=43, wid=14800)
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    _check_rows(o, lse, q, k, v, _rows(B, H, N, 12, seed=43), "bf16")


def test_long_head_backward():
    """B=1, H=1, N=16384, d=128, bf16: sampled rows of dQ, dK and dV against
    the oracle (whole-head forward in fp64 for O and LSE), sum identities."""
    B, H, N, d = 1, 1, 16384, 128
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=2.0, seed=44, wid=14900)
    do = make_dout(B, H, N, d, "bf16", seed=44, wid=14900)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, dc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    sv = dv.double().sum(dim=2)
    assert (sv - dc.double().sum(dim=2)).abs().max().item() <= 1e-2 * dv.double().abs().sum(dim=2).max().item()
    o_ref, lse_ref = oracle.attn(q, k, v)
    idx = sorted({i for _, _, i in _rows(B, H, N, 12, seed=44)})
    rows = [(0, 0, i) for i in idx]
    rq, rk, rv = oracle.attn_bwd_rows(q, k, v, o_ref, do, lse_ref, rows, rows)
    gate(dq[0, 0, idx].cpu().double().numpy(), rq, "dQ")
    gate(dk[0, 0, idx].cpu().double().numpy(), rk, "dK")
    gate(dv[0, 0, idx].cpu().double().numpy(), rv, "dV")
