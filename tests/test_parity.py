"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle.

Small and ragged shapes are compared element by element over every output,
and so are the two small workloads; the large ones are compared in full in
test_parity_whole.py.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from workloads import WORKLOADS, make_inputs, make_qkv, rising_norm_order

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.lib()


def run_gpu(q, k, v, scale=None):
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def check(q, k, v, dtype, scale=None, label=""):
    o, lse = run_gpu(q, k, v, scale)
    o_ref, lse_ref = oracle.attn(q, k, v, scale=scale)
    res = compare(o, lse, o_ref, lse_ref, dtype)
    assert res["ok"], f"{label} {res}"
    return res


SMALL = [
    # B, H, N, d, dtype, sigma_qk
    (1, 1, 1, 128, "bf16", 1.0),
    (1, 1, 63, 128, "f16", 1.0),
    (1, 2, 128, 128, "bf16", 1.0),
    (1, 1, 129, 128, "f16", 1.0),
    (2, 3, 200, 128, "bf16", 3.0),
    (1, 2, 256, 128, "f16", 1.0),
    (1, 1, 257, 128, "bf16", 1.0),
    (2, 2, 383, 128, "f16", 1.0),
    (1, 3, 700, 128, "bf16", 3.0),
    (1, 1, 1000, 128, "f16", 2.0),
    (1, 1, 1, 64, "f16", 1.0),
    (1, 1, 65, 64, "bf16", 1.0),
    (2, 2, 300, 64, "bf16", 3.0),
    (1, 1, 777, 64, "f16", 1.0),
    (4, 33, 64, 64, "f16", 1.0),
]


@pytest.mark.parametrize("B,H,N,d,dtype,sig", SMALL, ids=lambda x: str(x))
def test_small_shapes(B, H, N, d, dtype, sig):
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=11, wid=1000 + N + d)
    check(q, k, v, dtype, label=f"{B}x{H}x{N}x{d} {dtype}")


SMALL_F32 = [
    # B, H, N, d
    (1, 1, 1, 64),
    (1, 2, 100, 64),
    (1, 3, 129, 64),
    (2, 1, 300, 128),
    (1, 1, 33, 128),
    (1, 1, 257, 128),
]


@pytest.mark.parametrize("B,H,N,d", SMALL_F32, ids=lambda x: str(x))
def test_f32_shapes(B, H, N, d):
    q, k, v = make_qkv(B, H, N, d, "f32", seed=13, wid=6000 + N + d)
    check(q, k, v, "f32", label=f"{B}x{H}x{N}x{d} f32")


def test_f32_rescale_stress():
    """sigma 3 makes every score 9 times larger than with unit inputs, so the
    error of any fp32 evaluation of the scores (and of O and LSE through exp)
    grows 9 times too; the fp32 gates are scaled by sigma^2 = 9 here."""
    q, k, v = make_qkv(1, 2, 400, 64, "f32", sigma_qk=3.0, seed=2, wid=6100)
    k, v = rising_norm_order(k, v)
    o, lse = run_gpu(q, k, v)
    o_ref, lse_ref = oracle.attn(q, k, v)
    assert np.abs(o - o_ref).max() <= 9 * 1e-5
    assert np.all(np.abs(lse - lse_ref) <= 9 * (1e-5 + 1e-6 * np.abs(lse_ref)))


@pytest.mark.parametrize("N", [128, 384])
@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f16")])
def test_single_kv_tile_and_exact_multiples(N, d, dtype):
    q, k, v = make_qkv(1, 2, N, d, dtype, seed=5, wid=2000 + N)
    check(q, k, v, dtype)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (128, "f16"), (64, "bf16")])
def test_rescale_stress_rising_key_norms(d, dtype):
    """Keys sorted by rising norm with sigma 3: the row max grows on most tiles."""
    q, k, v = make_qkv(1, 2, 1024, d, dtype, sigma_qk=3.0, seed=9, wid=3000 + d)
    k, v = rising_norm_order(k, v)
    check(q, k, v, dtype)


@pytest.mark.parametrize("tau", [0.0, 8.0, 15.0])
@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (128, "f16"), (64, "bf16"), (256, "bf16")])
def test_rescale_stress_threshold_eager_and_lazy(d, dtype, tau):
    """The rising-norm sigma-3 stress through the testing build with the
    rescale threshold set to 0 (O rescaled whenever a row's max grows, as the
    dataflow page's section 2.3 describes), to 8 and to the default 15 (log2
    units): all meet the gates, element by element."""
    from exact_attention_87_gb300 import testing
    q, k, v = make_qkv(1, 2, 1024, d, dtype, sigma_qk=3.0, seed=9, wid=3100 + d)
    k, v = rising_norm_order(k, v)
    o, lse, _ = testing.attention_debug(q.cuda(), k.cuda(), v.cuda(), tau=tau)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, dtype)
    assert res["ok"], f"tau={tau} {res}"


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f16")])
def test_fp32_output_small_shapes_strict_gate(d, dtype):
    """fa_fwd_debug's fp32 output on ragged shapes: raw 1e-2 against the oracle."""
    from exact_attention_87_gb300 import testing
    from parity_util import TOL
    q, k, v = make_qkv(2, 3, 700, d, dtype, sigma_qk=3.0, seed=10, wid=3200 + d)
    o32, lse, _ = testing.attention_debug(q.cuda(), k.cuda(), v.cuda(), out_f32=True)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    o_ref, lse_ref = oracle.attn(q, k, v)
    err = np.abs(o32.cpu().double().numpy() - o_ref)
    assert err.max() <= 1e-2, err.max()
    lerr = np.abs(lse.cpu().double().numpy() - lse_ref)
    assert np.all(lerr <= TOL[dtype]["lse_rel"] * np.maximum(1.0, np.abs(lse_ref)))


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (4, 40, 1024, 64, "bf16"),    # 640 units on one CTA per SM: four or five per CTA
    (3, 52, 1024, 64, "f16"),
    (3, 52, 1024, 128, "f16"),
])
def test_persistent_several_units_per_cta(B, H, N, d, dtype):
    """The persistent form (d = 64 and 128, N a multiple of 256): each CTA
    walks several units with the barrier phases carried across them; every
    output against the oracle, keys in rising-norm order with sigma 3 so
    that rows rescale across units' boundaries too."""
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=3.0, seed=12, wid=4100 + N + d + H)
    k, v = rising_norm_order(k, v)
    check(q, k, v, dtype)


def test_non_default_scale():
    q, k, v = make_qkv(1, 2, 300, 128, "bf16", seed=3, wid=4000)
    check(q, k, v, "bf16", scale=0.3)


@pytest.mark.parametrize("name", ["b1h1n64d64_f32", "b1h4n512d64_f16"])
def test_whole_small_workloads(name):
    """The two small workloads fit the oracle in full: every output is compared."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    check(q, k, v, w.dtype, label=w.name)


def test_deterministic():
    q, k, v = make_qkv(2, 4, 1000, 128, "bf16", sigma_qk=3.0, seed=1, wid=5000)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.attention(qc, kc, vc)
    o1, l1 = o1.clone(), l1.clone()
    for _ in range(5):
        o2, l2 = fa.attention(qc, kc, vc)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def sample_rows(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    edge = [0, 1, 127, 128, 255, 256, N - 1, N - 2, N // 2]
    for t in range(n):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        i = edge[t] if t < len(edge) else int(rng.integers(N))
        if 0 <= i < N:
            rows.add((b, h, i))
    return sorted(rows)
