"""The order in which the backward's main kernels take key tiles, and the
one-CTA-per-unit forward kernels their work units (no GPU).

Definition (include/fa_testing.h, fa_testing_bwd_tile): CTA c of the
B*H*ceil(N/128) CTAs takes one (b*h, key tile). Without the causal mask a
head's key tiles come in a row (c = bh * nt + kt). With the causal mask key
tile kt visits nt - kt Q tiles, and the CTAs are dealt out longest first
within windows of W heads, W = clamp(64 MiB // (8 N d), 1, B*H): window w
holds heads [w W, w W + g) with g = min(W, B*H - w W), and within it
position j (c = w W nt + j) takes key tile j // g of head w W + j % g. The
tests rebuild that order here and read the library's copy of the device
arithmetic back through fa_testing_bwd_tile.
"""
import pytest

from exact_attention_87_gb300 import testing as fat


def expected(B, H, N, d, causal):
    nt = -(-N // 128)
    bhn = B * H
    if not causal:
        return [(bh, kt) for bh in range(bhn) for kt in range(nt)]
    W = max(1, min(bhn, (64 << 20) // (8 * N * d)))
    order = []
    for h0 in range(0, bhn, W):
        g = min(W, bhn - h0)
        for kt in range(nt):
            order += [(h0 + x, kt) for x in range(g)]
    return order


SHAPES = [
    (8, 32, 4096, 128),   # 16 heads a window
    (8, 32, 4096, 64),    # 32
    (4, 16, 4096, 256),   # 8
    (1, 3, 4096, 128),    # one partial window
    (2, 9, 1000, 128),    # ragged N: 8 key tiles, W = 18 (all heads)
    (3, 7, 16384, 128),   # 4 heads a window, the last window 1 head
    (1, 1, 1, 64),        # one CTA
    (5, 5, 131072, 256),  # W = 1: the causal order is the plain one
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_backward_tile_order_matches_the_definition(B, H, N, d, causal):
    want = expected(B, H, N, d, causal)
    ctas = len(want)
    # every CTA for small grids; a spread of CTAs (ends, window edges) for large ones
    idx = range(ctas) if ctas <= 4096 else sorted({*range(0, ctas, 97), *range(ctas - 300, ctas), *range(300)})
    for c in idx:
        rc, got = fat.bwd_tile(B, H, N, d, causal, c)
        assert rc == 1 and got == want[c], (c, got, want[c])
    # the definition itself is a permutation of all (head, key tile) pairs
    assert sorted(want) == [(bh, kt) for bh in range(B * H) for kt in range(-(-N // 128))]


def test_causal_windows_put_long_key_tiles_first():
    """Within a window every head's key tile t comes before any head's key
    tile t + 1, so the CTAs of a window run longest first (key tile t visits
    nt - t Q tiles)."""
    B, H, N, d = 8, 32, 4096, 128
    order = expected(B, H, N, d, True)
    W, nt = 16, 32
    for w in range(B * H // W):
        win = order[w * W * nt:(w + 1) * W * nt]
        kts = [kt for _, kt in win]
        assert kts == sorted(kts)
        assert {bh for bh, _ in win} == set(range(w * W, (w + 1) * W))


def test_backward_tile_argument_errors():
    assert fat.bwd_tile(0, 1, 128, 128, 0, 0)[0] == -1
    assert fat.bwd_tile(1, 1, 128, 96, 0, 0)[0] == -1
    assert fat.bwd_tile(1, 1, 128, 128, 0, 1)[0] == -1      # one key tile: CTA 1 does not exist
    assert fat.bwd_tile(1, 1, 128, 128, 1, -1)[0] == -1
    assert fat.bwd_tile(65536, 65536, 4096, 128, 0, 0)[0] == -1   # 2^37 CTAs


# ---------------------------------------------------------------------------
# The forward's one-CTA-per-unit kernels (fa_testing_fwd_unit): unit u of an
# unsplit launch over every unit takes one (b*h, Q block). Without the causal
# mask a head's Q blocks come in a row (u = bh * nqb + qb). With it, Q block
# qb sees qb + 1 blocks' worth of keys, and units are dealt out longest first
# within windows of W heads, W = clamp(64 MiB // (4 N d), 1, B*H): window w
# holds heads [w W, w W + g), g = min(W, B*H - w W), and its position j takes
# Q block nqb - 1 - j // g of head w W + j % g; a launch whose units all fit
# on the device's SMs at once (num_sms > 0, units <= num_sms) takes them
# longest first within each head (u -> head u // nqb, block nqb - 1 - u % nqb).
# ---------------------------------------------------------------------------
def expected_fwd(B, H, N, d, causal, num_sms=0):
    rows = 128 if d == 256 else 256
    nqb = -(-N // rows)
    bhn = B * H
    if not causal:
        return [(bh, qb) for bh in range(bhn) for qb in range(nqb)]
    if 0 < num_sms and bhn * nqb <= num_sms:
        return [(bh, nqb - 1 - qb) for bh in range(bhn) for qb in range(nqb)]
    W = max(1, min(bhn, (64 << 20) // (4 * N * d)))
    order = []
    for h0 in range(0, bhn, W):
        g = min(W, bhn - h0)
        for j in range(nqb):
            order += [(h0 + x, nqb - 1 - j) for x in range(g)]
    return order


FWD_SHAPES = [
    (8, 32, 4096, 128),   # 32 heads a window (the persistent kernel takes this shape; the order is the fallback's)
    (1, 8, 16384, 128),   # 8 heads: all in one window
    (8, 32, 4096, 64),    # 64
    (4, 16, 4096, 256),   # 16 heads, 128-row Q tiles
    (3, 7, 1000, 128),    # ragged N, all 21 heads in one window
    (2, 3, 65536, 128),   # 2 heads a window, the last window 2
    (1, 1, 1, 64),
]


@pytest.mark.parametrize("num_sms", [0, 152])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", FWD_SHAPES + [(1, 4, 512, 64), (2, 19, 1024, 128)])
def test_forward_unit_order_matches_the_definition(B, H, N, d, causal, num_sms):
    want = expected_fwd(B, H, N, d, causal, num_sms)
    n = len(want)
    idx = range(n) if n <= 4096 else sorted({*range(0, n, 89), *range(n - 300, n), *range(300)})
    for u in idx:
        rc, got = fat.fwd_unit(B, H, N, d, causal, u, num_sms)
        assert rc == 1 and got == want[u], (u, got, want[u])
    rows = 128 if d == 256 else 256
    assert sorted(want) == [(bh, qb) for bh in range(B * H) for qb in range(-(-N // rows))]


def test_forward_unit_argument_errors():
    assert fat.fwd_unit(0, 1, 256, 128, 0, 0)[0] == -1
    assert fat.fwd_unit(1, 1, 256, 96, 0, 0)[0] == -1
    assert fat.fwd_unit(1, 1, 256, 128, 1, 1)[0] == -1     # one 256-row block: unit 1 does not exist
    assert fat.fwd_unit(1, 1, 256, 256, 1, 1)[0] == 1      # two 128-row tiles at d = 256
    assert fat.fwd_unit(1, 1, 256, 128, 0, -1)[0] == -1
    assert fat.fwd_unit(1, 1, 256, 128, 0, 0, -1)[0] == -1  # negative SM count
