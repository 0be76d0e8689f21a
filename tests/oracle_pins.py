"""Pins for the CPU oracle: checks against facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an oracle library handle and raises AssertionError when the
oracle disagrees with something that does not depend on the oracle itself:
hand-derived worked examples, closed forms, invariants, brute force on tiny
inputs, and library routines (numpy/scipy) for the textbook special case.
``tests/test_oracle.py`` runs them against the real oracle, and against
builds with one planted mistake each, which must fail at least one pin.
"""
import itertools
import math

import numpy as np

import oracle
from golden_cases import all_cases

RNG = np.random.default_rng(1234)


def _attn(lib, q, k, v, scale=None, nthreads=2):
    return oracle.attn(q, k, v, scale=scale, nthreads=nthreads, lib=lib)


def pin_golden(lib):
    """Hand-derived worked examples (tests/golden)."""
    for c in all_cases():
        o, lse = _attn(lib, c["Q"], c["K"], c["V"], scale=c["scale"])
        np.testing.assert_allclose(o, c["O"], rtol=0, atol=c["tol"], err_msg=c["name"])
        np.testing.assert_allclose(lse, c["LSE"], rtol=0, atol=c["tol"], err_msg=c["name"])


def pin_brute_force(lib):
    """Tiny inputs against sums of exp of the raw scores (no max shift), exact-summed."""
    rng = np.random.default_rng(7)
    for Nq, Nk, d in [(1, 1, 1), (2, 3, 2), (3, 4, 3), (4, 2, 5), (3, 3, 1)]:
        q, k, v = (rng.standard_normal((n, d)) for n in (Nq, Nk, Nk))
        scale = 0.7
        o, lse = _attn(lib, q, k, v, scale=scale)
        for i in range(Nq):
            s = [scale * math.fsum(q[i, c] * k[j, c] for c in range(d)) for j in range(Nk)]
            w = [math.exp(x) for x in s]
            Z = math.fsum(w)
            for c in range(d):
                ref = math.fsum(w[j] * v[j, c] for j in range(Nk)) / Z
                assert abs(o[i, c] - ref) <= 1e-13 * max(1.0, abs(ref)), (Nq, Nk, d, i, c)
            assert abs(lse[i] - math.log(Z)) <= 1e-13 * max(1.0, abs(math.log(Z)))


def pin_rows_sum_to_one(lib):
    """With V = identity (Nk = d) the output rows are the softmax rows: >= 0, sum 1."""
    for N, scale in [(8, 0.5), (33, 0.2), (64, 1.0 / 8)]:
        q, k = RNG.standard_normal((2, 3, N, N)), RNG.standard_normal((2, 3, N, N))
        v = np.broadcast_to(np.eye(N), (2, 3, N, N)).copy()
        p, _ = _attn(lib, q, k, v, scale=scale)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)


def pin_zero_query(lib):
    """Q = 0: every score is 0, P is uniform, O = column mean of V, LSE = ln Nk."""
    for Nq, Nk, d in [(5, 7, 3), (4, 64, 16), (1, 129, 8)]:
        q = np.zeros((Nq, d))
        k, v = RNG.standard_normal((Nk, d)) * 3, RNG.standard_normal((Nk, d))
        o, lse = _attn(lib, q, k, v, scale=0.3)
        np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, math.log(Nk), rtol=0, atol=1e-13)


def pin_identical_keys(lib):
    """All keys equal: P is uniform, O = mean of V, LSE = scale q.k + ln Nk."""
    Nq, Nk, d, scale = 6, 40, 5, 0.4
    q = RNG.standard_normal((Nq, d))
    key = RNG.standard_normal(d)
    k = np.broadcast_to(key, (Nk, d)).copy()
    v = RNG.standard_normal((Nk, d))
    o, lse = _attn(lib, q, k, v, scale=scale)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=0, atol=1e-13)
    expect = np.array([scale * math.fsum(q[i] * key) + math.log(Nk) for i in range(Nq)])
    np.testing.assert_allclose(lse, expect, rtol=0, atol=1e-12)


def pin_constant_v_column(lib):
    """A V column that is constant c passes through as c (convex combination)."""
    Nq, Nk, d = 9, 23, 4
    q, k = RNG.standard_normal((Nq, d)) * 2, RNG.standard_normal((Nk, d)) * 2
    v = RNG.standard_normal((Nk, d))
    v[:, 2] = -3.25
    o, _ = _attn(lib, q, k, v, scale=0.9)
    np.testing.assert_allclose(o[:, 2], -3.25, rtol=1e-14, atol=0)


def pin_shift_invariance(lib):
    """K <- K + 1 w^T adds scale*q.w to a whole score row: O unchanged, LSE += scale*q.w."""
    B, H, N, d, scale = 2, 2, 31, 6, 0.35
    q, k, v = (RNG.standard_normal((B, H, N, d)) for _ in range(3))
    w = RNG.standard_normal(d) * 2
    o0, l0 = _attn(lib, q, k, v, scale=scale)
    o1, l1 = _attn(lib, q, k + w, v, scale=scale)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0 + scale * (q @ w), rtol=0, atol=1e-12)


def pin_permutation(lib):
    """Joint K/V row permutation leaves O, LSE unchanged; a Q row permutation permutes them."""
    N, d = 17, 5
    q, k, v = (RNG.standard_normal((1, 2, N, d)) for _ in range(3))
    o0, l0 = _attn(lib, q, k, v, scale=0.5)
    pk = RNG.permutation(N)
    o1, l1 = _attn(lib, q, k[:, :, pk], v[:, :, pk], scale=0.5)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-13)
    pq = RNG.permutation(N)
    o2, l2 = _attn(lib, q[:, :, pq], k, v, scale=0.5)
    np.testing.assert_allclose(o2, o0[:, :, pq], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l0[:, :, pq], rtol=0, atol=1e-13)


def pin_head_independence(lib):
    """A batched call equals one call per (batch, head)."""
    B, H, Nq, Nk, d = 2, 3, 7, 11, 4
    q = RNG.standard_normal((B, H, Nq, d))
    k, v = RNG.standard_normal((B, H, Nk, d)), RNG.standard_normal((B, H, Nk, d))
    o, lse = _attn(lib, q, k, v, scale=0.6, nthreads=3)
    for b, h in itertools.product(range(B), range(H)):
        o1, l1 = _attn(lib, q[b, h], k[b, h], v[b, h], scale=0.6, nthreads=1)
        np.testing.assert_array_equal(o[b, h], o1)
        np.testing.assert_array_equal(lse[b, h], l1)


def pin_hard_attention_limit(lib):
    """Integer scores with a unique row max and scale 60: P is one-hot to < e^-60."""
    Nq, Nk, d = 6, 9, 3
    rng = np.random.default_rng(5)
    while True:
        q = rng.integers(-3, 4, (Nq, d)).astype(float)
        k = rng.integers(-3, 4, (Nk, d)).astype(float)
        s = q @ k.T
        top = np.sort(s, axis=1)
        if np.all(top[:, -1] - top[:, -2] >= 1):
            break
    v = rng.standard_normal((Nk, d))
    o, lse = _attn(lib, q, k, v, scale=60.0)
    np.testing.assert_allclose(o, v[s.argmax(1)], rtol=0, atol=1e-20 + 1e-24)
    np.testing.assert_allclose(lse, 60.0 * s.max(1), rtol=1e-15, atol=1e-12)


def pin_single_key(lib):
    """Nk = 1: P = 1, O = v, LSE = s."""
    q, k, v = RNG.standard_normal((5, 4)), RNG.standard_normal((1, 4)), RNG.standard_normal((1, 4))
    o, lse = _attn(lib, q, k, v, scale=0.25)
    np.testing.assert_array_equal(o, np.broadcast_to(v[0], o.shape))
    np.testing.assert_allclose(lse, 0.25 * (q @ k[0]), rtol=0, atol=1e-14)


def pin_linearity_in_v(lib):
    """O is linear in V for fixed Q, K."""
    Nq, Nk, d = 8, 19, 5
    q, k = RNG.standard_normal((Nq, d)), RNG.standard_normal((Nk, d))
    v1, v2 = RNG.standard_normal((Nk, d)), RNG.standard_normal((Nk, d))
    o1, _ = _attn(lib, q, k, v1, scale=0.5)
    o2, _ = _attn(lib, q, k, v2, scale=0.5)
    o3, _ = _attn(lib, q, k, v1 - 2.5 * v2, scale=0.5)
    np.testing.assert_allclose(o3, o1 - 2.5 * o2, rtol=0, atol=1e-12)


def pin_library_reference(lib):
    """Textbook special case through library routines: scipy softmax/logsumexp of q @ k.T."""
    from scipy.special import logsumexp, softmax
    for B, H, Nq, Nk, d in [(1, 2, 37, 53, 16), (2, 1, 64, 64, 64), (1, 1, 130, 257, 8)]:
        q = RNG.standard_normal((B, H, Nq, d)) * 1.5
        k, v = RNG.standard_normal((B, H, Nk, d)) * 1.5, RNG.standard_normal((B, H, Nk, d))
        scale = 1.0 / math.sqrt(d)
        s = np.einsum("bhid,bhjd->bhij", q, k) * scale
        o_ref = np.einsum("bhij,bhjd->bhid", softmax(s, axis=-1), v)
        o, lse = _attn(lib, q, k, v, scale=scale)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, logsumexp(s, axis=-1), rtol=0, atol=1e-11)


def pin_large_magnitude(lib):
    """Scores of order +-1000 stay finite and obey the shift rule against a small copy."""
    Nq, Nk, d = 4, 12, 3
    q = RNG.standard_normal((Nq, d))
    k = RNG.standard_normal((Nk, d))
    v = RNG.standard_normal((Nk, d))
    w = np.array([300.0, -200.0, 500.0])
    o0, l0 = _attn(lib, q, k, v, scale=1.0)
    o1, l1 = _attn(lib, q, k + w, v, scale=1.0)  # scores shift by q.w, several hundred
    assert np.all(np.isfinite(o1)) and np.all(np.isfinite(l1))
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(l1, l0 + q @ w, rtol=1e-14, atol=1e-10)


def _bwd(lib, q, k, v, w, scale):
    """Gradients of L = sum(W * O) from the oracle (dO = W), with the oracle's own O and LSE."""
    o, lse = _attn(lib, q, k, v, scale=scale)
    return oracle.attn_bwd(q, k, v, o, w, lse, scale=scale, nthreads=2, lib=lib)


def pin_bwd_finite_differences(lib):
    """Backward pass against central differences of the forward oracle's L = sum(W * O)."""
    rng = np.random.default_rng(11)
    B, H, N, d, scale = 1, 2, 9, 5, 0.6
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    w = rng.standard_normal((B, H, N, d))
    dq, dk, dv = _bwd(lib, q, k, v, w, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (0, 0, 8, 4), (0, 1, 3, 1), (0, 0, 5, 3)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            lp = float((w * _attn(lib, *args_p, scale=scale)[0]).sum())
            lm = float((w * _attn(lib, *args_m, scale=scale)[0]).sum())
            assert abs((lp - lm) / (2 * h) - g[idx]) <= 1e-7 * max(1.0, abs(g[idx])), (name, idx)


def pin_bwd_invariants(lib):
    """Rows of P sum to one, so sum_j dV_j = sum_i dO_i; O does not change under
    K -> K + 1 w^T, so sum_j dK_j = 0; O is linear in V, so V -> 3V leaves dV
    and triples dQ and dK."""
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((2, 2, 33, 8)) * 1.5 for _ in range(3))
    w = rng.standard_normal(q.shape)
    dq, dk, dv = _bwd(lib, q, k, v, w, 0.35)
    np.testing.assert_allclose(dv.sum(axis=2), w.sum(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    dq2, dk2, dv2 = _bwd(lib, q, k, 3.0 * v, w, 0.35)
    np.testing.assert_allclose(dv2, dv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq2, 3.0 * dq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk2, 3.0 * dk, rtol=1e-12, atol=1e-12)


def pin_bwd_single_key(lib):
    """N = 1: O = v whatever q and k are, so dV = dO and dQ = dK = 0."""
    rng = np.random.default_rng(13)
    q, k, v, w = (rng.standard_normal((1, 1, 1, 4)) for _ in range(4))
    dq, dk, dv = _bwd(lib, q, k, v, w, 0.5)
    np.testing.assert_allclose(dv, w, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


def pin_bwd_uniform_attention(lib):
    """Q = 0: P = 1/N everywhere, so dV_j = mean_i dO_i, and the closed form
    dQ_i = scale/N * sum_j (dO_i . (v_j - O_i)) k_j with O_i = mean_j v_j."""
    rng = np.random.default_rng(14)
    N, d, scale = 7, 3, 0.8
    q = np.zeros((1, 1, N, d))
    k, v, w = (rng.standard_normal((1, 1, N, d)) for _ in range(3))
    dq, dk, dv = _bwd(lib, q, k, v, w, scale)
    np.testing.assert_allclose(dv[0, 0], np.broadcast_to(w[0, 0].mean(0), (N, d)), rtol=0, atol=1e-14)
    vbar = v[0, 0].mean(0)
    for i in range(N):
        ref = np.zeros(d)
        for j in range(N):
            ref += math.fsum(w[0, 0, i] * (v[0, 0, j] - vbar)) * k[0, 0, j]
        np.testing.assert_allclose(dq[0, 0, i], scale / N * ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0 * dk, atol=1e-13)  # q_i = 0 multiplies every term


def pin_bwd_masked_finite_differences(lib):
    """Masked backward (causal, key lengths, both, and a batch with no key at
    all) against central differences of the masked forward's L = sum(W * O)."""
    rng = np.random.default_rng(15)
    B, H, N, d, scale = 3, 2, 8, 4, 0.7
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    w = rng.standard_normal((B, H, N, d))
    h = 1e-6
    for causal, klen in ((True, None), (False, [8, 5, 0]), (True, [3, 8, 6])):
        o, lse = oracle.attn_masked(q, k, v, causal=causal, klen=klen, scale=scale, nthreads=2, lib=lib)
        dq, dk, dv = oracle.attn_bwd(q, k, v, o, w, lse, scale=scale, nthreads=2, lib=lib, causal=causal,
                                     klen=klen)

        def loss(qq, kk, vv):
            oo = oracle.attn_masked(qq, kk, vv, causal=causal, klen=klen, scale=scale, nthreads=2, lib=lib)[0]
            return float((w * oo).sum())

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (1, 0, 7, 3), (1, 1, 5, 1), (2, 0, 2, 0), (2, 1, 6, 3),
                        (1, 0, 4, 2), (0, 0, 7, 1)]:
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                ap = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                am = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                fd = (loss(*ap) - loss(*am)) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(g[idx])), (causal, klen, name, idx)


def pin_bwd_masked_structure(lib):
    """Causal row 0 sees only key 0 (O_0 = v_0), so dQ_0 = 0 and the last key
    is seen only by the last query; keys at or past a batch's length get zero
    dK and dV, and a batch with no key gets zero gradients everywhere."""
    rng = np.random.default_rng(16)
    B, H, N, d, scale = 2, 2, 10, 3, 0.9
    q, k, v, w = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    o, lse = oracle.attn_masked(q, k, v, causal=True, scale=scale, nthreads=2, lib=lib)
    dq, dk, dv = oracle.attn_bwd(q, k, v, o, w, lse, scale=scale, nthreads=2, lib=lib, causal=True)
    np.testing.assert_allclose(dq[:, :, 0], 0.0, atol=1e-15)
    last = N - 1
    p_last = np.exp(scale * np.einsum("bhc,bhc->bh", q[:, :, last], k[:, :, last]) - lse[:, :, last])
    np.testing.assert_allclose(dv[:, :, last], p_last[..., None] * w[:, :, last], rtol=1e-12, atol=1e-14)
    klen = [6, 0]
    o, lse = oracle.attn_masked(q, k, v, klen=klen, scale=scale, nthreads=2, lib=lib)
    dq, dk, dv = oracle.attn_bwd(q, k, v, o, w, lse, scale=scale, nthreads=2, lib=lib, klen=klen)
    assert np.all(dk[0, :, 6:] == 0.0) and np.all(dv[0, :, 6:] == 0.0)
    assert np.all(dq[1] == 0.0) and np.all(dk[1] == 0.0) and np.all(dv[1] == 0.0)
    # the unmasked keys obey the unmasked invariant: sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv[0].sum(axis=1), w[0].sum(axis=1), rtol=0, atol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
