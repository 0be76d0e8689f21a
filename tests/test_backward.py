"""GPU parity of the backward pass (fa_bwd, through the C ABI) against the CPU fp64 oracle.

The GPU backward takes the GPU forward's O and LSE, as a training step would;
the oracle takes its own fp64 forward results. Small and ragged shapes are
compared over every element of dQ, dK and dV; the full-size workload runs in
the benchmark's configuration and is compared on sampled rows of sampled heads,
plus sum identities that hold for every head.

Gate (per gradient tensor): max |g - g_ref| <= 1e-2 * max |g_ref| and cosine
similarity >= 0.999 (a reference that is 0, as dQ and dK are with a single
key, must come out below 1e-3 in magnitude). Rounding P and dS*scale to 8 significant bits (bf16)
before the products, as the kernel does, gives 0.3-0.6 % of max |g_ref| on
these inputs in an fp64 model of those roundings; the gradients grow with the
input scale (sigma^2 for dQ and dK), hence a gate relative to max |g_ref|.
"""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from workloads import WORKLOADS, make_dout, make_inputs, make_qkv, rising_norm_order

pytestmark = pytest.mark.gpu

REL_TOL = 1e-2
COS_TOL = 0.999


@pytest.fixture(scope="module", autouse=True)
def _cuda_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.lib()


ZERO_FLOOR = 1e-3  # a gradient that is exactly 0 (dQ, dK with one key) must come out below this


def gate(got, ref, label):
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{label}: non-finite values"
    err = np.abs(got - ref).max()
    mx = np.abs(ref).max()
    if mx < ZERO_FLOOR:
        assert np.abs(got).max() <= ZERO_FLOOR, f"{label}: reference ~0 (max {mx:.3e}), got max {np.abs(got).max():.3e}"
        return err, 1.0
    cos = float((got * ref).sum() / np.sqrt((got * got).sum() * (ref * ref).sum()))
    assert err <= REL_TOL * mx and cos >= COS_TOL, f"{label}: max err {err:.3e} (max ref {mx:.3e}) cos {cos:.6f}"
    return err / mx, cos


def gpu_fwd_bwd(q, k, v, do, scale=None):
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, dc, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return [t.cpu().double().numpy() for t in (dq, dk, dv)]


def check(B, H, N, d, dtype, sig=1.0, seed=3, wid=8000, scale=None, order=False):
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=seed, wid=wid)
    if order:
        k, v = rising_norm_order(k, v)
    do = make_dout(B, H, N, d, dtype, seed=seed, wid=wid)
    got = gpu_fwd_bwd(q, k, v, do, scale)
    o, lse = oracle.attn(q, k, v, scale=scale)
    ref = oracle.attn_bwd(q, k, v, o, do, lse, scale=scale)
    return [gate(g, r, f"{n} {B}x{H}x{N}x{d} {dtype}") for n, g, r in zip(("dQ", "dK", "dV"), got, ref)]


SMALL = [
    # B, H, N, d, dtype, sigma_qk
    (1, 1, 1, 128, "bf16", 1.0),
    (1, 1, 1, 64, "f16", 1.0),
    (1, 2, 128, 128, "bf16", 1.0),
    (1, 1, 129, 128, "f16", 1.0),
    (2, 3, 200, 128, "bf16", 2.0),
    (1, 2, 256, 64, "bf16", 1.0),
    (1, 1, 257, 64, "f16", 1.0),
    (2, 2, 383, 128, "f16", 1.0),
    (1, 2, 640, 128, "bf16", 3.0),
    (1, 1, 1000, 64, "bf16", 2.0),
    (3, 5, 64, 64, "f16", 1.0),
    # d = 256: two main kernels, 64-row Q tiles
    (1, 1, 1, 256, "bf16", 1.0),
    (1, 2, 128, 256, "bf16", 1.0),
    (1, 1, 129, 256, "f16", 1.0),
    (2, 2, 300, 256, "bf16", 2.0),
    (1, 2, 640, 256, "bf16", 3.0),
    (2, 1, 1000, 256, "f16", 1.0),
]


@pytest.mark.parametrize("B,H,N,d,dtype,sig", SMALL, ids=lambda x: str(x))
def test_backward_small_shapes(B, H, N, d, dtype, sig):
    check(B, H, N, d, dtype, sig, wid=8000 + N + d)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f16"), (256, "bf16")])
def test_backward_rising_key_norms(d, dtype):
    """sigma 3 with keys sorted by norm: sharply peaked rows, P near 0 and 1."""
    check(1, 2, 768, d, dtype, 3.0, wid=8100 + d, order=True)


@pytest.mark.parametrize("d", [128, 256])
def test_backward_non_default_scale(d):
    check(1, 2, 300, d, "bf16", 1.0, wid=8200, scale=0.3)


@pytest.mark.parametrize("d", [128, 256])
def test_backward_deterministic(d):
    """dK and dV are written once per key tile; dQ is a sum of fp32 reduce-adds
    over key tiles, whose order can vary: it must agree to fp32 rounding."""
    q, k, v = (t.cuda() for t in make_qkv(1, 4, 700, d, "bf16", sigma_qk=2.0, seed=1, wid=8300))
    do = make_dout(1, 4, 700, d, "bf16", seed=1, wid=8300).cuda()
    o, lse = fa.attention(q, k, v)
    ref = [t.clone() for t in fa.attention_backward(q, k, v, o, lse, do)]
    for _ in range(3):
        dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do)
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


@pytest.mark.parametrize("B,H,N,d,dtype", [(4, 20, 512, 128, "bf16"), (3, 16, 768, 64, "f16"), (2, 41, 256, 128, "f16")])
def test_backward_more_key_tiles_than_sms(B, H, N, d, dtype):
    """320, 288 and 164 key tiles: more CTAs than a 152-SM device holds at once
    (one CTA per SM), so later waves start on SMs whose previous CTA left TMEM,
    barriers and shared memory behind."""
    check(B, H, N, d, dtype, 2.0, wid=8450 + N + d)


@pytest.mark.parametrize("B,H,N,d", [(4, 20, 512, 128), (3, 16, 768, 64), (8, 32, 4096, 128)])
def test_backward_full_tile_instantiation_matches_the_masked_one(B, H, N, d):
    """With no mask and N a multiple of 128 the backward runs the instantiation
    that compiles only the unmasked copy of the P loop; a key-length array of
    all N selects the masked instantiation, in which nothing is masked. Both
    compute each key tile's products in the same order: dK and dV must be
    bit-identical, dQ (fp32 reduce-adds in a varying order) equal to fp32
    rounding. The last shape is the benchmark's workload."""
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, "bf16", sigma_qk=3.0, seed=5, wid=8500 + d))
    do = make_dout(B, H, N, d, "bf16", seed=5, wid=8500 + d).cuda()
    o, lse = fa.attention(q, k, v)
    a = fa.attention_backward(q, k, v, o, lse, do)
    kl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    b = fa.attention_backward(q, k, v, o, lse, do, seqlens_k=kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    err = (a[0].float() - b[0].float()).abs().max().item()
    assert err <= 1e-2 * b[0].float().abs().max().item()


def test_backward_reuses_workspace_and_outputs():
    """A caller workspace and preallocated outputs holding garbage give the same result."""
    B, H, N, d = 1, 2, 300, 64
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, "bf16", seed=2, wid=8400))
    do = make_dout(B, H, N, d, "bf16", seed=2, wid=8400).cuda()
    o, lse = fa.attention(q, k, v)
    ref = fa.attention_backward(q, k, v, o, lse, do)
    ws = torch.full((fa.fa_bwd_workspace_size(B, H, N, d),), 0x7F, dtype=torch.uint8, device="cuda")
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]
    got = fa.attention_backward(q, k, v, o, lse, do, dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    # dQ: fp32 reduce-adds in an order that can vary, rounded once
    assert (got[0].float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


def test_backward_full_workload_sampled():
    """The benchmark workload (B=8, H=32, N=4096, d=128, bf16, sigma 3): sampled
    rows of three heads against the oracle, sum identities for every head."""
    w = WORKLOADS["b8h32n4096d128_bf16_qk3"]
    q, k, v = make_inputs(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, dc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    # Identities of every head: rows of P sum to 1, so sum_j dV_j = sum_i dO_i;
    # O is unchanged by K -> K + 1 w^T, so sum_j dK_j = 0.
    sv = dv.double().sum(dim=2)
    assert (sv - dc.double().sum(dim=2)).abs().max().item() <= 1e-2 * dv.double().abs().sum(dim=2).max().item()
    sk = dk.double().sum(dim=2)
    assert sk.abs().max().item() <= 1e-2 * dk.double().abs().sum(dim=2).max().item()
    # Sampled rows of three heads against the oracle (whole-head forward for O, LSE).
    rng = np.random.default_rng(w.wid)
    heads = [(0, 0), (3, 17), (7, 31)]
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        qh, kh, vh, dh = (t[sl] for t in (q, k, v, do))
        oh, lh = oracle.attn(qh, kh, vh)
        idx = sorted({0, 1, 127, 128, w.N - 1, *rng.integers(0, w.N, 27).tolist()})
        rows = [(0, 0, i) for i in idx]
        rq, rk, rv = oracle.attn_bwd_rows(qh, kh, vh, oh, dh, lh, rows, rows)
        gq = dq[b, h, idx].cpu().double().numpy()
        gk = dk[b, h, idx].cpu().double().numpy()
        gv = dv[b, h, idx].cpu().double().numpy()
        gate(gq, rq, f"dQ head {b},{h}")
        gate(gk, rk, f"dK head {b},{h}")
        gate(gv, rv, f"dV head {b},{h}")


def test_backward_d256_workload_sampled():
    """The head-dimension-256 workload (B=4, H=16, N=4096, bf16): sampled rows
    of two heads against the oracle, sum identities for every head."""
    w = WORKLOADS["b4h16n4096d256_bf16"]
    q, k, v = make_inputs(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention(qc, kc, vc)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, dc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    sv = dv.double().sum(dim=2)
    assert (sv - dc.double().sum(dim=2)).abs().max().item() <= 1e-2 * dv.double().abs().sum(dim=2).max().item()
    sk = dk.double().sum(dim=2)
    assert sk.abs().max().item() <= 1e-2 * dk.double().abs().sum(dim=2).max().item()
    rng = np.random.default_rng(w.wid)
    for b, h in [(0, 0), (3, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        qh, kh, vh, dh = (t[sl] for t in (q, k, v, do))
        oh, lh = oracle.attn(qh, kh, vh)
        idx = sorted({0, 1, 63, 64, 127, 128, w.N - 1, *rng.integers(0, w.N, 25).tolist()})
        rows = [(0, 0, i) for i in idx]
        rq, rk, rv = oracle.attn_bwd_rows(qh, kh, vh, oh, dh, lh, rows, rows)
        gate(dq[b, h, idx].cpu().double().numpy(), rq, f"dQ head {b},{h}")
        gate(dk[b, h, idx].cpu().double().numpy(), rk, f"dK head {b},{h}")
        gate(dv[b, h, idx].cpu().double().numpy(), rv, f"dV head {b},{h}")
