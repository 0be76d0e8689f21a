"""GPU parity of the masked backward pass (fa_bwd_ex: causal mask, per-batch
key lengths) against the CPU fp64 oracle's masked backward.

The GPU forward runs with the same masks (fa_fwd_ex) and hands its O and LSE
to the backward, as a training step would; the oracle uses its own masked
forward. The gate is the one of the unmasked backward tests (max error within
1e-2 of max |g_ref|, cosine >= 0.999). Masked keys must get exactly zero dK and
dV, and a batch with no key at all exactly zero gradients: there the masked
products are exact zeros, not small numbers.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from workloads import WORKLOADS, make_dout, make_inputs, make_qkv

pytestmark = pytest.mark.gpu

REL_TOL = 1e-2
COS_TOL = 0.999
ZERO_FLOOR = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.lib()


def gate(got, ref, label):
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{label}: non-finite values"
    err = np.abs(got - ref).max()
    mx = np.abs(ref).max()
    if mx < ZERO_FLOOR:
        assert np.abs(got).max() <= ZERO_FLOOR, f"{label}: reference ~0 (max {mx:.3e}), got max {np.abs(got).max():.3e}"
        return
    cos = float((got * ref).sum() / np.sqrt((got * got).sum() * (ref * ref).sum()))
    assert err <= REL_TOL * mx and cos >= COS_TOL, f"{label}: max err {err:.3e} (max ref {mx:.3e}) cos {cos:.6f}"


def run(q, k, v, do, causal, klen, scale=None):
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    kl = None if klen is None else torch.tensor(klen, dtype=torch.int32, device="cuda")
    o, lse = fa.attention(qc, kc, vc, scale=scale, causal=causal, seqlens_k=kl)
    grads = fa.attention_backward(qc, kc, vc, o, lse, dc, scale=scale, causal=causal, seqlens_k=kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return [t.cpu().double().numpy() for t in grads]


def check(B, H, N, d, dtype, causal, klen, sig=1.0, wid=8600, scale=None, pad_value=None):
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=5, wid=wid)
    do = make_dout(B, H, N, d, dtype, seed=5, wid=wid)
    if pad_value is not None and klen is not None:
        # masked keys and values hold large finite garbage: it must not reach the gradients
        for b, n in enumerate(klen):
            n = min(max(n, 0), N)
            k[b, :, n:] = pad_value
            v[b, :, n:] = -pad_value
    got = run(q, k, v, do, causal, klen, scale)
    o, lse = oracle.attn_masked(q, k, v, causal=causal, klen=klen, scale=scale)
    ref = oracle.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=causal, klen=klen)
    label = f"{B}x{H}x{N}x{d} {dtype} causal={causal} klen={klen}"
    for n, g, r in zip(("dQ", "dK", "dV"), got, ref):
        gate(g, r, f"{n} {label}")
    if klen is not None:
        for b, n in enumerate(klen):
            n = min(max(n, 0), N)
            assert np.all(got[1][b, :, n:] == 0.0) and np.all(got[2][b, :, n:] == 0.0), f"masked keys {label}"
            if n == 0:
                assert np.all(got[0][b] == 0.0), f"dQ of a batch with no key {label}"


CAUSAL = [
    # B, H, N, d, dtype, sigma_qk
    (1, 1, 1, 128, "bf16", 1.0),
    (1, 2, 128, 128, "bf16", 1.0),
    (1, 1, 129, 64, "f16", 1.0),
    (2, 3, 200, 128, "bf16", 2.0),
    (1, 1, 257, 64, "f16", 1.0),
    (2, 2, 383, 128, "f16", 1.0),
    (1, 2, 640, 128, "bf16", 3.0),
    (1, 1, 1000, 64, "bf16", 2.0),
    (1, 1, 65, 256, "bf16", 1.0),
    (2, 2, 300, 256, "bf16", 2.0),
    (1, 1, 640, 256, "f16", 1.0),
]


@pytest.mark.parametrize("B,H,N,d,dtype,sig", CAUSAL, ids=lambda x: str(x))
def test_causal_backward(B, H, N, d, dtype, sig):
    check(B, H, N, d, dtype, True, None, sig, wid=8600 + N + d)


KLEN = [
    # B, H, N, d, dtype, causal, key lengths (0 = no key; past N or negative are clamped)
    (3, 2, 300, 128, "bf16", False, [300, 128, 0]),
    (3, 2, 300, 64, "f16", False, [129, 1, 299]),
    (2, 3, 513, 128, "bf16", False, [1000, -4]),
    (3, 2, 300, 128, "f16", True, [300, 200, 0]),
    (2, 2, 640, 64, "bf16", True, [257, 640]),
    (3, 2, 300, 256, "bf16", False, [300, 64, 0]),
    (2, 2, 333, 256, "f16", True, [200, 333]),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,klen", KLEN, ids=lambda x: str(x))
def test_key_length_backward(B, H, N, d, dtype, causal, klen):
    check(B, H, N, d, dtype, causal, klen, 1.5, wid=8700 + N + d)


def test_padded_keys_hold_garbage():
    check(2, 2, 400, 128, "bf16", False, [150, 333], 1.0, wid=8800, pad_value=1.0e4)
    check(2, 2, 400, 64, "f16", True, [150, 333], 1.0, wid=8801, pad_value=1.0e3)


def test_causal_non_default_scale():
    check(1, 2, 300, 128, "bf16", True, None, 1.0, wid=8810, scale=0.3)


def test_masked_backward_deterministic_dk_dv():
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 700, 128, "bf16", sigma_qk=2.0, seed=6, wid=8820))
    do = make_dout(2, 4, 700, 128, "bf16", seed=6, wid=8820).cuda()
    kl = torch.tensor([700, 333], dtype=torch.int32, device="cuda")
    o, lse = fa.attention(q, k, v, causal=True, seqlens_k=kl)
    ref = [t.clone() for t in fa.attention_backward(q, k, v, o, lse, do, causal=True, seqlens_k=kl)]
    for _ in range(3):
        dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=True, seqlens_k=kl)
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


def test_causal_full_workload_sampled():
    """The benchmark workload (B=8, H=32, N=4096, d=128, bf16, sigma 3) with the
    causal mask: sampled rows of three heads against the oracle, and the
    identity sum_j dV_j = sum_i dO_i (each row's P sums to 1 over the keys it sees)."""
    w = WORKLOADS["b8h32n4096d128_bf16_qk3"]
    q, k, v = make_inputs(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, causal=True)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, dc, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    sv = dv.double().sum(dim=2)
    assert (sv - dc.double().sum(dim=2)).abs().max().item() <= 1e-2 * dv.double().abs().sum(dim=2).max().item()
    rng = np.random.default_rng(w.wid + 1)
    for b, h in [(0, 0), (4, 9), (7, 31)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        qh, kh, vh, dh = (t[sl] for t in (q, k, v, do))
        oh, lh = oracle.attn_masked(qh, kh, vh, causal=True)
        idx = sorted({0, 1, 127, 128, w.N - 1, *rng.integers(0, w.N, 27).tolist()})
        rows = [(0, 0, i) for i in idx]
        rq, rk, rv = oracle.attn_bwd_rows(qh, kh, vh, oh, dh, lh, rows, rows, causal=True)
        gate(dq[b, h, idx].cpu().double().numpy(), rq, f"dQ head {b},{h}")
        gate(dk[b, h, idx].cpu().double().numpy(), rk, f"dK head {b},{h}")
        gate(dv[b, h, idx].cpu().double().numpy(), rv, f"dV head {b},{h}")
