"""Head dimension 256 (fp16 / bf16 forward pass): GPU parity against the CPU
fp64 oracle over every output, with masks, plus the MMA issue-order check."""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from exact_attention_87_gb300 import _build
from parity_util import compare
from workloads import make_qkv, rising_norm_order

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.lib()


def run(q, k, v, scale=None, causal=False, klen=None):
    kl = torch.tensor(klen, dtype=torch.int32, device="cuda") if klen is not None else None
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, seqlens_k=kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def check(q, k, v, dtype, scale=None, causal=False, klen=None, label=""):
    o, lse = run(q, k, v, scale, causal, klen)
    if causal or klen is not None:
        o_ref, lse_ref = oracle.attn_masked(q, k, v, causal=causal, klen=klen, scale=scale)
    else:
        o_ref, lse_ref = oracle.attn(q, k, v, scale=scale)
    empty = np.isneginf(lse_ref)
    assert np.all(o[empty] == 0) and np.all(np.isneginf(lse[empty]))
    res = compare(o[~empty], lse[~empty], o_ref[~empty], lse_ref[~empty], dtype)
    assert res["ok"], f"{label} {res}"


@pytest.mark.parametrize("B,H,N,dtype,sig", [
    (1, 1, 1, "bf16", 1.0),
    (1, 1, 63, "f16", 1.0),
    (1, 2, 64, "bf16", 1.0),
    (1, 1, 65, "f16", 1.0),
    (1, 2, 128, "bf16", 2.0),
    (2, 3, 200, "bf16", 3.0),
    (1, 2, 257, "f16", 1.0),
    (2, 1, 700, "bf16", 1.0),
    (1, 1, 1000, "f16", 2.0),
])
def test_d256_shapes(B, H, N, dtype, sig):
    q, k, v = make_qkv(B, H, N, 256, dtype, sigma_qk=sig, seed=51, wid=14000 + N)
    check(q, k, v, dtype, label=f"{B}x{H}x{N}x256 {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_d256_rescale_stress(dtype):
    q, k, v = make_qkv(1, 2, 1024, 256, dtype, sigma_qk=3.0, seed=52, wid=14100)
    k, v = rising_norm_order(k, v)
    check(q, k, v, dtype)


def test_d256_non_default_scale():
    q, k, v = make_qkv(1, 2, 300, 256, "bf16", seed=53, wid=14200)
    check(q, k, v, "bf16", scale=0.11)


@pytest.mark.parametrize("B,H,N,dtype", [(1, 2, 1000, "bf16"), (2, 1, 321, "f16")])
def test_d256_causal(B, H, N, dtype):
    q, k, v = make_qkv(B, H, N, 256, dtype, sigma_qk=2.0, seed=54, wid=14300 + N)
    check(q, k, v, dtype, causal=True)


def test_d256_key_lengths_and_causal():
    q, k, v = make_qkv(4, 2, 500, 256, "bf16", seed=55, wid=14400)
    check(q, k, v, "bf16", klen=[500, 1, 64, 0])
    check(q, k, v, "bf16", causal=True, klen=[500, 130, 65, 0])


def test_d256_fp32_is_refused():
    q = torch.zeros((1, 1, 64, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.attention(q, q, q)
    assert e.value.code == fa.FA_ERR_HEADDIM


def test_d256_default_order_equals_strict_order():
    """S_{j+2} is issued right behind P_j V_j, whose P it overwrites; the strict
    build waits for P_j V_j instead. Same MMAs in the same order: bit-identical."""
    L = ctypes.CDLL(_build.build(strict=True))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    L.fa_fwd.restype = i
    B, H, N, d = 2, 8, 2048, 256
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, "bf16", sigma_qk=3.0, seed=56, wid=14500))
    o1, l1 = fa.attention(q, k, v)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    rc = L.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), B, H, N, d,
                  1.0 / d ** 0.5, fa.FA_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
