"""CPU tests of the oracle: pins, the online recurrence model, and planted mistakes."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle_pins
from workloads import WORKLOADS, make_inputs, make_qkv


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# Each mutant plants one plausible mistake in the oracle source (see ORACLE_MUTANT
# in oracle/attn_ref.c); at least one pin must catch it.
MUTANTS = {
    1: "wrong component index in q.k",
    2: "scale dropped",
    3: "row max not subtracted",
    4: "sign error in the exponent",
    5: "off-by-one value row",
    6: "max term dropped from LSE",
    7: "transposed score matrix",
    8: "backward: D term dropped from dS",
    9: "backward: scale dropped from dK",
    10: "backward: P transposed in dV",
    11: "backward: causal mask off by one",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    path = oracle.build(out=str(tmp_path / f"liboracle_m{mutant}.so"), mutant=mutant)
    lib = oracle.load(path)
    assert lib.oracle_mutant_id() == mutant
    caught = []
    with np.errstate(all="ignore"):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(lib)
            except (AssertionError, FloatingPointError, ValueError, RuntimeError):
                caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"


def test_real_oracle_is_not_a_mutant(oracle_lib):
    assert oracle_lib.oracle_mutant_id() == 0


# ---- online recurrence model (tiled formula of the MUSA guide) vs the definition ----

@pytest.mark.parametrize("block_n", [1, 16, 64, 128])
@pytest.mark.parametrize("tau", [0.0, 8 * np.log(2.0)])
def test_online_equals_three_pass(block_n, tau):
    for (B, H, N, d, sig) in [(1, 2, 200, 16, 1.0), (1, 1, 512, 64, 3.0), (2, 1, 129, 8, 3.0)]:
        q, k, v = make_qkv(B, H, N, d, "f32", sigma_qk=sig, seed=3, wid=90 + block_n)
        o3, l3 = oracle.attn(q, k, v)
        o1, l1 = oracle.attn_online(q, k, v, block_n=block_n, tau=tau)
        np.testing.assert_allclose(o1, o3, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1, l3, rtol=0, atol=1e-12)


def test_online_trace_ends_at_lse():
    """The last block's running (m, l) gives LSE = m + ln l; m never decreases."""
    q, k, v = make_qkv(1, 2, 96, 32, "f32", sigma_qk=3.0, seed=1, wid=77)
    o, lse, tm, tl = oracle.attn_online(q, k, v, block_n=16, tau=0.0, trace=True)
    np.testing.assert_allclose(tm[..., -1] + np.log(tl[..., -1]), lse, rtol=0, atol=1e-12)
    assert np.all(np.diff(tm, axis=-1) >= 0)
    # eager (tau = 0): after every block m equals the max of the scores seen so far
    qd, kd = q.double().numpy(), k.double().numpy()
    s = np.einsum("bhid,bhjd->bhij", qd, kd) / np.sqrt(32)
    for b in range(tm.shape[-1]):
        np.testing.assert_allclose(tm[..., b], s[..., : 16 * (b + 1)].max(-1), rtol=0, atol=1e-12)


def test_lazy_rescale_moves_reference_less_often():
    """With tau = 8 ln 2 the reference max moves on fewer blocks than with tau = 0."""
    q, k, v = make_qkv(1, 1, 512, 64, "f32", sigma_qk=3.0, seed=2, wid=78)
    _, _, m0, _ = oracle.attn_online(q, k, v, block_n=64, tau=0.0, trace=True)
    _, _, m8, _ = oracle.attn_online(q, k, v, block_n=64, tau=8 * np.log(2.0), trace=True)
    moves0 = (np.diff(m0, axis=-1) > 0).sum()
    moves8 = (np.diff(m8, axis=-1) > 0).sum()
    assert moves8 < moves0


def test_rows_api_matches_full():
    q, k, v = make_qkv(2, 2, 70, 16, "bf16", seed=0, wid=55)
    o, lse = oracle.attn(q, k, v)
    rows = [(0, 0, 0), (1, 1, 69), (0, 1, 33), (1, 0, 5)]
    ro, rl = oracle.attn_rows(q, k, v, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], o[b, h, i], rtol=0, atol=1e-15)
        np.testing.assert_allclose(rl[n], lse[b, h, i], rtol=0, atol=1e-15)


# ---- seeded input generator ----

def test_inputs_are_deterministic_and_rounded():
    w = WORKLOADS["b1h4n512d64_f16"]
    a = make_inputs(w)
    b = make_inputs(w)
    for x, y in zip(a, b):
        assert x.dtype == y.dtype and x.is_contiguous()
        assert bool((x == y).all())
    assert a[0].shape == (1, 4, 512, 64)
    qk3 = make_qkv(1, 2, 256, 128, "bf16", sigma_qk=3.0, sigma_v=1.0, seed=0, wid=4)
    assert 2.5 < float(qk3[0].float().std()) < 3.5
    assert 0.8 < float(qk3[2].float().std()) < 1.2


# ---- block merge (split-KV) ----

@pytest.mark.parametrize("cuts", [[0, 700], [0, 128, 700], [0, 1, 300, 301, 700], [0, 350, 351, 700]])
def test_merge_of_key_ranges_equals_whole(cuts):
    """Attention over disjoint key ranges, merged, equals attention over all keys."""
    q, k, v = make_qkv(2, 2, 700, 32, "f32", sigma_qk=3.0, seed=6, wid=120)
    o_ref, l_ref = oracle.attn(q, k, v)
    parts = [oracle.attn(q, k[:, :, a:b], v[:, :, a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = oracle.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, rtol=0, atol=1e-12)


def test_merge_special_cases():
    rng = np.random.default_rng(3)
    o1, l1 = rng.standard_normal((5, 4)), rng.standard_normal(5) * 10
    o, lse = oracle.merge(o1[None], l1[None])            # one part: identity
    np.testing.assert_array_equal(o, o1)
    np.testing.assert_allclose(lse, l1, rtol=0, atol=1e-15)
    o, lse = oracle.merge(np.stack([o1, o1]), np.stack([l1, l1]))   # two equal parts: same O, LSE + ln 2
    np.testing.assert_allclose(o, o1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, l1 + np.log(2.0), rtol=0, atol=1e-14)
    o2 = rng.standard_normal((5, 4))
    o, lse = oracle.merge(np.stack([o1, o2]), np.stack([l1, l1 - 800.0]))  # a negligible part
    np.testing.assert_allclose(o, o1, rtol=0, atol=1e-300 + 1e-15)
    # order of the parts does not matter
    oa, la = oracle.merge(np.stack([o1, o2]), np.stack([l1, l1 - 1.0]))
    ob, lb = oracle.merge(np.stack([o2, o1]), np.stack([l1 - 1.0, l1]))
    np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-14)


# ---- masks: causal and per-batch key lengths ----

def test_masked_without_masks_is_the_definition():
    q, k, v = make_qkv(2, 3, 70, 16, "bf16", seed=2, wid=130)
    o0, l0 = oracle.attn(q, k, v)
    o1, l1 = oracle.attn_masked(q, k, v)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_causal_rows_are_prefix_attention():
    """Causal row i equals unmasked attention of q_i over keys 0..i (brute force)."""
    q, k, v = make_qkv(1, 2, 40, 8, "f32", sigma_qk=2.0, seed=3, wid=131)
    o, lse = oracle.attn_masked(q, k, v, causal=True)
    for i in [0, 1, 7, 20, 39]:
        oi, li = oracle.attn(q[:, :, i:i + 1], k[:, :, : i + 1], v[:, :, : i + 1])
        np.testing.assert_allclose(o[:, :, i], oi[:, :, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], li[:, :, 0], rtol=0, atol=1e-13)
    # row 0 sees only key 0: O = v_0, LSE = s_00
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    np.testing.assert_allclose(o[:, :, 0], vd[:, :, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], (qd[:, :, 0] * kd[:, :, 0]).sum(-1) / np.sqrt(8), rtol=0, atol=1e-13)
    # the last row sees every key
    o_full, l_full = oracle.attn(q, k, v)
    np.testing.assert_allclose(o[:, :, -1], o_full[:, :, -1], rtol=0, atol=1e-13)


def test_key_lengths_equal_truncated_keys():
    q, k, v = make_qkv(3, 2, 50, 8, "f32", seed=4, wid=132)
    klen = [50, 17, 1]
    o, lse = oracle.attn_masked(q, k, v, klen=klen)
    for b, n in enumerate(klen):
        ob, lb = oracle.attn(q[b], k[b, :, :n], v[b, :, :n])
        np.testing.assert_allclose(o[b], ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], lb, rtol=0, atol=1e-13)
    # causal and key lengths together: row i sees keys j < min(i + 1, klen[b])
    o2, l2 = oracle.attn_masked(q, k, v, causal=True, klen=klen)
    for b, n in enumerate(klen):
        for i in [0, 5, 30, 49]:
            m = min(i + 1, n)
            oi, li = oracle.attn(q[b, :, i:i + 1], k[b, :, :m], v[b, :, :m])
            np.testing.assert_allclose(o2[b, :, i], oi[:, 0], rtol=0, atol=1e-13)


def test_fully_masked_rows_are_guarded():
    """No allowed key: O = 0 and LSE = -inf, never NaN."""
    q, k, v = make_qkv(2, 1, 20, 8, "f32", seed=5, wid=133)
    o, lse = oracle.attn_masked(q, k, v, klen=[0, 20])
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(o[1])) and np.all(np.isfinite(lse[1]))



def test_backward_rows_match_full_backward(oracle_lib):
    """The sampled-row backward (used at full sizes) against the full backward."""
    rng = np.random.default_rng(21)
    B, H, N, d, scale = 2, 2, 37, 8, 0.4
    q, k, v, w = (rng.standard_normal((B, H, N, d)) * 1.3 for _ in range(4))
    o, lse = oracle.attn(q, k, v, scale=scale)
    dq, dk, dv = oracle.attn_bwd(q, k, v, o, w, lse, scale=scale)
    rows = [(0, 0, 0), (1, 1, 36), (0, 1, 17), (1, 0, 5)]
    rq, rk, rv = oracle.attn_bwd_rows(q, k, v, o, w, lse, rows, rows[::-1], scale=scale)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(rq[n], dq[b, h, i], rtol=0, atol=1e-14)
    for n, (b, h, j) in enumerate(rows[::-1]):
        np.testing.assert_allclose(rk[n], dk[b, h, j], rtol=0, atol=1e-14)
        np.testing.assert_allclose(rv[n], dv[b, h, j], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal,klen", [(True, None), (False, [30, 0]), (True, [17, 37])])
def test_masked_backward_rows_match_full_backward(oracle_lib, causal, klen):
    """The sampled-row backward with masks against the full masked backward."""
    rng = np.random.default_rng(22)
    B, H, N, d, scale = 2, 2, 37, 8, 0.4
    q, k, v, w = (rng.standard_normal((B, H, N, d)) * 1.3 for _ in range(4))
    o, lse = oracle.attn_masked(q, k, v, causal=causal, klen=klen, scale=scale)
    dq, dk, dv = oracle.attn_bwd(q, k, v, o, w, lse, scale=scale, causal=causal, klen=klen)
    rows = [(0, 0, 0), (1, 1, 36), (0, 1, 17), (1, 0, 5), (0, 0, 29), (0, 1, 30), (1, 1, 16)]
    rq, rk, rv = oracle.attn_bwd_rows(q, k, v, o, w, lse, rows, rows[::-1], scale=scale, causal=causal, klen=klen)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(rq[n], dq[b, h, i], rtol=0, atol=1e-14)
    for n, (b, h, j) in enumerate(rows[::-1]):
        np.testing.assert_allclose(rk[n], dk[b, h, j], rtol=0, atol=1e-14)
        np.testing.assert_allclose(rv[n], dv[b, h, j], rtol=0, atol=1e-14)
