"""The default MMA issue order against the strictly ordered build, bit for bit.

P_i(j) lives in the tensor-memory columns of S_i, and the default build issues
S_i(j+1) right behind P_i(j) V_j, relying on one CTA's MMAs executing in issue
order. The strict build (-DFA_STRICT_MMA_ORDER) instead waits for P_i(j) V_j
to complete. Both run the same MMAs with the same accumulation order, so their
outputs must be identical bit for bit; any overwrite of P before it was read
would show up as a difference.
"""
import ctypes

import pytest
import torch

import exact_attention_87_gb300 as fa
from exact_attention_87_gb300 import _build
from workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def strict_lib():
    L = ctypes.CDLL(_build.build(strict=True))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    L.fa_fwd.restype = i
    L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, vp]
    L.fa_fwd_ex.restype = i
    return L


@pytest.mark.parametrize("B,H,N,d,dtype,sig,causal", [
    (2, 16, 4096, 128, "bf16", 3.0, False),   # the persistent form: 512 units on one CTA per SM
    (2, 16, 4096, 128, "bf16", 3.0, True),    # its causal form: heavy/light pairs
    (2, 16, 4096, 64, "f16", 1.0, False),     # its d = 64 form (stages freed by commits)
    (1, 8, 8192, 128, "f16", 1.0, False),
    (4, 8, 1000, 64, "bf16", 1.0, False),
    (3, 5, 777, 128, "f16", 2.0, False),
])
def test_default_order_equals_strict_order(strict_lib, B, H, N, d, dtype, sig, causal):
    """The product build (S issued right behind the P.V that reads its
    columns; the persistent form where it applies) against the strict-order
    build (one CTA per unit, every P.V waited for): bit for bit."""
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=21, wid=9000 + N))
    o1, l1 = fa.attention(q, k, v, causal=causal)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    code = fa.FA_BF16 if dtype == "bf16" else fa.FA_F16
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        rc = strict_lib.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                                  B, H, N, d, 1.0 / d ** 0.5, code, int(causal), None, stream)
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        o1, l1 = fa.attention(q, k, v, causal=causal)


@pytest.mark.parametrize("B,H,N,d,dtype,sig", [
    (1, 16, 2048, 128, "bf16", 3.0),
    (2, 4, 1000, 64, "f16", 1.0),
    (1, 3, 777, 128, "f16", 2.0),
    (1, 4, 1000, 256, "bf16", 2.0),   # the d = 256 dV kernel issues S^T_{i+2} behind dV_i
])
def test_backward_default_order_equals_strict_order(strict_lib, B, H, N, d, dtype, sig):
    """The backward kernel issues S^T_{i+2} behind dV_{i+1}, whose P^T it
    overwrites; the strict build waits for dV_{i+1} first. dK and dV (written
    once per key tile, same MMAs in the same order) must match bit for bit.
    dQ is a sum of fp32 reduce-adds whose order differs between runs anyway."""
    from workloads import make_dout
    vp, i, f, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
    strict_lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, u64, vp]
    strict_lib.fa_bwd.restype = i
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=22, wid=9100 + N))
    do = make_dout(B, H, N, d, dtype, seed=22, wid=9100 + N).cuda()
    o, lse = fa.attention(q, k, v)
    dq1, dk1, dv1 = fa.attention_backward(q, k, v, o, lse, do)
    dq2, dk2, dv2 = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    code = fa.FA_BF16 if dtype == "bf16" else fa.FA_F16
    rc = strict_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                           dq2.data_ptr(), dk2.data_ptr(), dv2.data_ptr(), B, H, N, d, 1.0 / d ** 0.5, code,
                           ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2 * dq1.float().abs().max().item()
