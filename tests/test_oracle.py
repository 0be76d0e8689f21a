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
