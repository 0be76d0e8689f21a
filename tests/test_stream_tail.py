"""The streamed tail of the persistent d = 128 forward, on the host (no GPU).

The units left over after the last full round of SMs are laid end to end as
K/V tiles and cut into one contiguous range per CTA (range c = [floor(c T /
G), floor((c + 1) T / G)) of the T tail tiles over G CTAs, the definition
include/fa.h gives for fa_fwd_stream_plan). A unit a range boundary cuts is
computed in pieces that are merged afterwards; the split into pieces is the
split-KV of the Triton page (section 2.3), with the cut points set by the
ranges. These tests check the library's own copy of the device arithmetic
(fa_testing_stream_piece) against that definition, written out here from it:
every tail tile belongs to exactly one piece, the pieces of a range are its
tiles in order, a piece is whole exactly when it covers its unit, part slots
are unique, and the merge finds exactly the pieces of each cut unit. Then the
plan queries: when the tail is streamed, and what the split-KV plan reports.
"""
import pytest

import exact_attention_87_gb300 as fa
from exact_attention_87_gb300 import testing as fat


def ranges(T, G):
    """The ranges of the definition: [floor(c T / G), floor((c + 1) T / G))."""
    return [(c * T // G, (c + 1) * T // G) for c in range(G)]


def pieces_of(T, G, n, c):
    """Pieces of range c read back through fa_testing_stream_piece, in order."""
    out = []
    for q in range(T + 2):
        rc, v = fat.stream_piece(T, G, n, c, q)
        assert rc in (0, 1)
        if rc == 0:
            # no piece q: none after it either
            assert fat.stream_piece(T, G, n, c, q + 1)[0] == 0
            break
        out.append(tuple(v))
    return out


CASES = [
    (128, 76, 16), (128, 64, 16), (128, 126, 16), (128, 152, 16),   # 8 units of 16 tiles (B=8 H=12 N=2048)
    (7168, 126, 128), (7168, 152, 128),                            # 56 units of 128 tiles (B=1 H=8 N=16384)
    (1024, 126, 32), (4608, 152, 32), (5, 3, 5), (5, 7, 5), (1, 1, 1), (1, 4, 1), (12, 5, 3), (97, 13, 8),
]


@pytest.mark.parametrize("T,G,n", CASES)
def test_partition_matches_the_range_definition(T, G, n):
    owner = {}
    slots = {}
    for c, (a, b) in enumerate(ranges(T, G)):
        got = pieces_of(T, G, n, c)
        if a == b:
            assert got == []
            continue
        # the pieces are the range's tiles, in order, cut at unit boundaries
        x = a
        for q, (i, t0, t1, slot) in enumerate(got):
            assert i * n + t0 == x and 0 <= t0 < t1 <= n
            x = i * n + t1
            for t in range(i * n + t0, i * n + t1):
                assert t not in owner
                owner[t] = (c, q)
            whole = t0 == 0 and t1 == n
            assert (slot == -1) == whole
            if not whole:
                # only the first and the last piece of a range can cut a unit
                assert slot == (2 * c if q == 0 else 2 * c + 1)
                assert q == 0 or q == len(got) - 1
                assert slot not in slots
                slots[slot] = (i, t0, t1)
        assert x == b
    assert sorted(owner) == list(range(T))
    # the merge's view of each unit: exactly the ranges that hold its tiles
    for i in range(T // n):
        rc, (c_lo, c_hi) = fat.stream_piece(T, G, n, i, -1)
        assert rc == 1
        holders = sorted({owner[t][0] for t in range(i * n, (i + 1) * n)})
        assert holders[0] == c_lo and holders[-1] == c_hi
        nonempty = [c for c in range(c_lo, c_hi + 1) if ranges(T, G)[c][0] < ranges(T, G)[c][1]]
        assert nonempty == holders
        if c_lo != c_hi:
            # every piece of a cut unit sits in the slot the merge computes
            for c in holders:
                a = ranges(T, G)[c][0]
                slot = 2 * c if a >= i * n else 2 * c + 1
                assert slots[slot][0] == i
            covered = sorted(t for s, (u, t0, t1) in slots.items() if u == i for t in range(t0, t1))
            assert covered == list(range(n))


def test_partition_argument_checks():
    assert fat.stream_piece(0, 1, 1, 0, 0)[0] == -1
    assert fat.stream_piece(4, 0, 1, 0, 0)[0] == -1
    assert fat.stream_piece(4, 2, 0, 0, 0)[0] == -1
    assert fat.stream_piece(4, 2, 1, 2, 0)[0] == -1          # no range 2
    assert fat.stream_piece(4, 2, 2, 2, -1)[0] == -1         # no unit 2 (4 tiles, 2 per unit)
    assert fat.stream_piece(1 << 20, 1 << 12, 1, 0, 0)[0] == -1  # tiles * ctas >= 2^31


def unit_pieces(T, G, n):
    """Pieces per tail unit under the definition."""
    per = [set() for _ in range(T // n)]
    for c, (a, b) in enumerate(ranges(T, G)):
        for t in range(a, b):
            per[t // n].add(c)
    return [len(s) for s in per]


@pytest.mark.parametrize("B,H,N,num_sms", [
    (8, 12, 2048, 152),    # 768 units: 5 full rounds, 8 units (128 tiles) streamed
    (1, 20, 2048, 152),    # 160 units: 1 full round, 8 left
    (3, 7, 2048, 152),     # 168 units: 1 full round, 16 left
    (1, 2, 4096, 152),     # 32 units: no full round, all streamed
])
def test_stream_plan_on_the_host(B, H, N, num_sms):
    rc, sp = fa.fa_fwd_stream_plan(B, H, N, 128, num_sms)
    assert rc == fa.FA_OK
    units = B * H * N // 256
    n = N // 128
    assert 1 <= sp["ctas"] <= num_sms
    assert sp["unit0"] == (units // num_sms) * num_sms
    assert sp["tiles"] == (units - sp["unit0"]) * n
    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, 128, 0, num_sms)
    assert rc == fa.FA_OK
    assert p["launches"] == 2 and p["first_split_unit"] == sp["unit0"]
    assert p["splits"] == max(unit_pieces(sp["tiles"], sp["ctas"], n))
    assert p["workspace_bytes"] >= 2 * sp["ctas"] * 256 * (128 * 4 + 4)
    # the library's built-in scratch holds the slots
    assert 2 * sp["ctas"] * 256 * (128 * 4 + 4) + 256 <= 32 << 20  # FA_NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("B,H,N,d,num_sms", [
    (8, 32, 4096, 128, 152),   # 26.9 rounds: the last round is nearly full, streaming does not pay
    (8, 19, 4096, 128, 152),   # 2432 units: exact rounds, nothing left over
    (8, 12, 2000, 128, 152),   # N not a multiple of 256
    (8, 12, 2048, 64, 152),    # d = 64 has no persistent form
    (4, 16, 4096, 256, 152),   # nor d = 256
    (2, 3, 4096, 128, 152),    # 96 units of 32 tiles: the merge of ~220 pieces costs more than it saves
    (8, 12, 2048, 128, 148),   # 768 units on 148 SMs: 5.19 rounds, the 28 left over fill enough of the last
    (1, 8, 16384, 128, 152),   # N > 4096: one CTA per unit (the key-range tail plan)
])
def test_stream_plan_declines(B, H, N, d, num_sms):
    rc, sp = fa.fa_fwd_stream_plan(B, H, N, d, num_sms)
    assert rc == fa.FA_OK and sp == {"unit0": 0, "tiles": 0, "ctas": 0}
    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, d, 0, num_sms)
    assert p["launches"] in (1, 3) or p["first_split_unit"] == 0


def test_explicit_split_counts_never_stream():
    for ns in (1, 2, 4):
        rc, p = fa.fa_fwd_splitkv_plan(8, 12, 2048, 128, ns, 152)
        assert rc == fa.FA_OK
        assert p["launches"] == (1 if ns == 1 else 2) and (ns == 1 or p["first_split_unit"] == 0)


def test_stream_plan_argument_errors():
    import ctypes
    assert fa.fa_fwd_stream_plan(0, 1, 256, 128, 152)[0] == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_stream_plan(1, 1, 256, 128, 0)[0] == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_stream_plan(1, 1, 256, 96, 152)[0] == fa.FA_ERR_HEADDIM
    assert fa.fa_fwd_stream_plan(65536, 65536, 256, 128, 152)[0] == fa.FA_ERR_SHAPE
    assert fa.lib().fa_fwd_stream_plan(1, 1, 256, 128, 152, None, None, None) == fa.FA_ERR_NULL


def test_streamed_call_checks_its_workspace_in_dry_run():
    """The streamed path refuses a workspace one byte short of what the
    queries report, or misaligned, before anything is enqueued (testing
    build, dry run: placeholder addresses, nothing launched)."""
    L = fat.lib()
    B, H, N, d = 8, 12, 2048, 128
    rc, sp = fa.fa_fwd_stream_plan(B, H, N, d, 152)
    if sp["ctas"] == 0:
        pytest.skip("no streamed tail on this SM count")
    need = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 0)
    base = 1 << 40
    L.fa_testing_set_dry_run(1)
    try:
        args = (base, base, base, base, base, B, H, N, d, 0.088, fa.FA_F16, 0)
        rc = L.fa_fwd_splitkv(*args, base, need, None)
        if rc == fa.FA_ERR_ARCH or rc == fa.FA_ERR_CUDA:
            pytest.skip("no device to plan for")
        assert rc == fa.FA_OK
        assert L.fa_fwd_splitkv(*args, base, need - 1, None) == fa.FA_ERR_WORKSPACE
        assert L.fa_fwd_splitkv(*args, base + 16, need, None) == fa.FA_ERR_WORKSPACE
        assert L.fa_fwd_splitkv(*args, None, need, None) == fa.FA_ERR_WORKSPACE
    finally:
        L.fa_testing_set_dry_run(0)
