"""fa_fwd_splitkv_noalloc: split-KV without a caller workspace.

This entry point is for callers that must not allocate device memory while
they run (allocation-free real-time paths, plugins whose host forbids
cudaMalloc, code that cannot afford the device synchronisation an allocation
implies); its partial results live in the library's built-in 32 MiB scratch.
Its output must match fa_fwd_splitkv run with a caller workspace and the same
split count, on two calls in a row (the second reuses the scratch left by the
first). The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
from parity_util import TOL
from workloads import make_qkv

pytestmark = pytest.mark.gpu


def _run_with_workspace(q, k, v, splits):
    B, H, N, d = q.shape
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    code = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_F16
    rc = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                           d ** -0.5, code, splits, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.fa_strerror(rc)
    return o, lse


def _run_noalloc(q, k, v, splits):
    B, H, N, d = q.shape
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    code = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_F16
    rc = fa.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                   d, d ** -0.5, code, splits, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.fa_strerror(rc)
    return o, lse


@pytest.mark.parametrize("B,H,N,d,dtype,splits", [
    (1, 4, 2048, 128, "bf16", 2),
    (2, 2, 1000, 64, "f16", 4),
])
def test_noalloc_matches_workspace_entry_point_twice(B, H, N, d, dtype, splits):
    fa.build()
    tol = TOL[dtype]
    for call in range(2):
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, dtype, sigma_qk=2.0, seed=30 + call, wid=12000 + N))
        o_ref, l_ref = _run_with_workspace(q, k, v, splits)
        o, l = _run_noalloc(q, k, v, splits)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        assert float((o.double() - o_ref.double()).abs().max()) <= tol["o"]
        lse_bound = tol["lse_rel"] * torch.clamp(l_ref.double().abs(), min=1.0)
        assert bool(((l.double() - l_ref.double()).abs() <= lse_bound).all())
        assert bool(torch.isfinite(o).all())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape whose split-KV partials exceed the built-in scratch is refused
    with FA_ERR_SCRATCH_LIMIT, on real buffers of that shape (4 x 256 MiB), so
    that a regression of the size check could only compute, never touch
    memory that does not exist; a NULL pointer with the same shape is refused
    with FA_ERR_NULL, before the scratch is looked at."""
    fa.build()
    B, H, N, d, splits = 1, 64, 16384, 128, 4
    assert fa.fa_fwd_splitkv_workspace_size(B, H, N, d, splits) > (32 << 20)
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k, v, o = torch.zeros_like(q), torch.zeros_like(q), torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    rc = fa.fa_fwd_splitkv_noalloc(*ptrs, B, H, N, d, d ** -0.5, fa.FA_BF16, splits, None)
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in fa.fa_strerror(rc)
    rc = fa.fa_fwd_splitkv_noalloc(0, *ptrs[1:], B, H, N, d, d ** -0.5, fa.FA_BF16, splits, None)
    assert rc == fa.FA_ERR_NULL
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK


def test_noalloc_runs_the_automatic_plan_on_the_long_sequence_workload():
    """B=1, H=8, N=16384, d=128 with the automatic plan: the tail plan's
    partial buffers (the last wave's rows only) fit the built-in scratch, and
    the result equals the workspace entry point's bit for bit."""
    fa.build()
    B, H, N, d = 1, 8, 16384, 128
    need = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 0)
    assert need <= (32 << 20)
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, "bf16", sigma_qk=1.0, seed=33, wid=12500))
    o_ref, l_ref = _run_with_workspace(q, k, v, 0)
    o, l = _run_noalloc(q, k, v, 0)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    assert bool(torch.isfinite(o).all())
