"""The C ABI: the library builds, loads and exports every entry point that
include/fa.h declares; argument errors come back as codes before any launch.

The argument-error tests pass placeholder addresses. They call the testing
build of the library (same host code, compiled with -DFA_TESTING) with its
dry-run switch on, under which a call that gets past every check returns
FA_OK without enqueuing anything: a check that regressed shows up as a wrong
status code, never as a kernel launched on memory that does not exist."""
import os
import re

import pytest

import exact_attention_87_gb300 as fa
from exact_attention_87_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fa.lib()


def declared_functions(header=None):
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h") and (header is None or f == header):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_get_device_status" in names and "fa_strerror" in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions("fa.h"):
        assert hasattr(L, name), f"{name} declared in include/fa.h but not exported"


def test_testing_symbols_only_in_testing_library(L):
    import ctypes
    testing = ctypes.CDLL(_build.build(testing=True))
    names = declared_functions("fa_testing.h")
    assert "fa_fwd_testing" in names
    for name in names:
        assert hasattr(testing, name), f"{name} not exported by the testing library"
        assert not hasattr(L, name), f"{name} leaked into the product library"
    for name in declared_functions("fa.h"):
        assert hasattr(testing, name)


def test_every_header_is_covered():
    inc = os.path.join(ROOT, "include")
    assert sorted(f for f in os.listdir(inc) if f.endswith(".h")) == ["fa.h", "fa_testing.h"]


def test_strerror_and_version(L):
    assert fa.fa_abi_version() >= 100
    for code in range(0, 14):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown status"
    assert fa.fa_strerror(12345) == "unknown status"


A = 1 << 20  # a 16-byte aligned placeholder address (dry runs only: never dereferenced)


@pytest.fixture(scope="module")
def D():
    """The testing library with dry runs on (same entry points and argument types)."""
    from exact_attention_87_gb300 import testing
    lib = testing.lib()
    lib.fa_testing_set_dry_run(1)
    yield lib
    lib.fa_testing_set_dry_run(0)


@pytest.mark.parametrize("args,code", [
    ((0, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16), fa.FA_ERR_NULL),
    ((A, A, A, A, 0, 1, 1, 64, 64, 0.125, fa.FA_F16), fa.FA_ERR_NULL),
    ((A, A, A, A, A, 1, 1, 64, 64, 0.125, 7), fa.FA_ERR_DTYPE),
    ((A, A, A, A, A, 0, 1, 64, 64, 0.125, fa.FA_F16), fa.FA_ERR_SHAPE),
    ((A, A, A, A, A, 1, 1, 0, 64, 0.125, fa.FA_F16), fa.FA_ERR_SHAPE),
    ((A, A, A, A, A, 1, -3, 64, 64, 0.125, fa.FA_F16), fa.FA_ERR_SHAPE),
    ((A, A, A, A, A, 1, 1, 64, 96, 0.125, fa.FA_F16), fa.FA_ERR_HEADDIM),
    ((A, A, A, A, A, 1, 1, 64, 256, 0.125, fa.FA_F32), fa.FA_ERR_HEADDIM),
    ((A, A, A, A, A, 1, 1, 64, 512, 0.125, fa.FA_BF16), fa.FA_ERR_HEADDIM),
    ((A, A, A, A, A, 1, 1, 64, 192, 0.125, fa.FA_F16), fa.FA_ERR_HEADDIM),
    ((A, A, A, A, A, 1, 1, 64, 64, 0.0, fa.FA_F16), fa.FA_ERR_SCALE),
    ((A, A, A, A, A, 1, 1, 64, 64, float("nan"), fa.FA_F16), fa.FA_ERR_SCALE),
    ((A, A, A, A, A, 1, 1, 64, 64, -1.0, fa.FA_F16), fa.FA_ERR_SCALE),
    ((A + 8, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16), fa.FA_ERR_ALIGN),
    ((A, A, A, A + 2, A, 1, 1, 64, 64, 0.125, fa.FA_BF16), fa.FA_ERR_ALIGN),
    ((A, A, A, A, A + 2, 1, 1, 64, 64, 0.125, fa.FA_F32), fa.FA_ERR_ALIGN),
    ((A, A, A, A, A, 65536, 65536, 1 << 20, 128, 0.1, fa.FA_F16), fa.FA_ERR_SHAPE),
])
def test_argument_errors_return_before_launch(D, args, code):
    assert D.fa_fwd(*args, None) == code


def test_missing_library_raises(tmp_path):
    with pytest.raises(ImportError):
        fa.lib(str(tmp_path / "nope.so"))


def test_splitkv_workspace_size_formula(L, D):
    assert fa.fa_fwd_splitkv_workspace_size(1, 8, 16384, 128, 1) == 0
    rows = 1 * 8 * 16384 * 3
    o_bytes = (rows * 128 * 4 + 255) // 256 * 256
    assert fa.fa_fwd_splitkv_workspace_size(1, 8, 16384, 128, 3) == o_bytes + rows * 4
    # requests beyond the number of 128-key tiles are clamped: N = 300 has 3 tiles
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 300, 64, 9) == fa.fa_fwd_splitkv_workspace_size(1, 1, 300, 64, 3)
    assert fa.fa_fwd_splitkv_workspace_size(0, 1, 300, 64, 2) == 0
    assert D.fa_fwd_splitkv(0, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16, 2, A, 1 << 20, None) == fa.FA_ERR_NULL
    assert D.fa_fwd_splitkv(A, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16, -1, A, 1 << 20, None) == fa.FA_ERR_SHAPE
    # the allocation-free variant checks every argument before it looks at its scratch
    big = (1, 64, 16384, 128, 0.088, fa.FA_BF16, 4)
    assert D.fa_fwd_splitkv_noalloc(0, A, A, A, A, *big, None) == fa.FA_ERR_NULL
    assert D.fa_fwd_splitkv_noalloc(A, A, A, A + 2, A, *big, None) == fa.FA_ERR_ALIGN
    assert D.fa_fwd_splitkv_noalloc(A, A, A, A, A, 1, 64, 16384, 96, 0.088, fa.FA_BF16, 4, None) == \
        fa.FA_ERR_HEADDIM
    assert D.fa_fwd_splitkv_noalloc(A, A, A, A, A, 1, 64, 16384, 128, -1.0, fa.FA_BF16, 4, None) == fa.FA_ERR_SCALE


def test_splitkv_launch_count_argument_errors(L):
    assert fa.fa_fwd_splitkv_launches(0, 1, 64, 64, 0) == -fa.FA_ERR_SHAPE
    assert fa.fa_fwd_splitkv_launches(1, 1, 64, 64, -1) == -fa.FA_ERR_SHAPE
    assert fa.fa_fwd_splitkv_launches(1, 1, 64, 96, 0) == -fa.FA_ERR_HEADDIM


def test_masked_entry_point_argument_errors(D):
    assert D.fa_fwd_ex(A, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16, 2, None, None) == fa.FA_ERR_SHAPE
    assert D.fa_fwd_ex(0, A, A, A, A, 1, 1, 64, 64, 0.125, fa.FA_F16, 1, None, None) == fa.FA_ERR_NULL
    ws = fa.fa_bwd_workspace_size(1, 1, 64, 64)
    args = [A] * 6 + [A] * 3 + [1, 1, 64, 64, 0.125, fa.FA_F16]
    assert D.fa_bwd_ex(*args, 2, None, 1 << 24, ws, None) == fa.FA_ERR_SHAPE
    assert D.fa_bwd_ex(*args, -1, None, 1 << 24, ws, None) == fa.FA_ERR_SHAPE
    assert D.fa_bwd_ex(*([0] + args[1:]), 1, None, 1 << 24, ws, None) == fa.FA_ERR_NULL
    assert D.fa_bwd_ex(*args, 1, None, 0, ws, None) == fa.FA_ERR_WORKSPACE
    assert D.fa_bwd_ex(*(args[:12] + [96, 0.125, fa.FA_F16]), 1, None, 1 << 24, ws, None) == fa.FA_ERR_HEADDIM


def test_partial_and_merge_argument_errors(D):
    #                 Q  K  V  Op Lp B  H  Nq  Nk  d    scale  dtype
    ok = [A, A, A, A, A, 1, 1, 64, 64, 64, 0.125, fa.FA_BF16, None]
    def part(**kw):
        a = list(ok)
        for i, name in enumerate(["Q", "K", "V", "Op", "Lp", "B", "H", "Nq", "Nk", "d", "scale", "dtype"]):
            if name in kw:
                a[i] = kw[name]
        return D.fa_fwd_partial(*a)
    assert part(Q=0) == fa.FA_ERR_NULL
    assert part(Lp=0) == fa.FA_ERR_NULL
    assert part(dtype=fa.FA_F32) == fa.FA_ERR_UNSUPPORTED
    assert part(dtype=7) == fa.FA_ERR_DTYPE
    assert part(Nk=0) == fa.FA_ERR_SHAPE
    assert part(Nq=0) == fa.FA_ERR_SHAPE
    assert part(d=96) == fa.FA_ERR_HEADDIM
    assert part(scale=-1.0) == fa.FA_ERR_SCALE
    assert part(Op=A + 4) == fa.FA_ERR_ALIGN
    #                Op Lp P  O  L  B  H  N   d   dtype
    okm = [A, A, 2, A, A, 1, 1, 64, 64, fa.FA_F16, None]
    def merge(**kw):
        a = list(okm)
        for i, name in enumerate(["Op", "Lp", "P", "O", "L", "B", "H", "N", "d", "dtype"]):
            if name in kw:
                a[i] = kw[name]
        return D.fa_merge(*a)
    assert merge(Op=0) == fa.FA_ERR_NULL
    assert merge(P=0) == fa.FA_ERR_SHAPE
    assert merge(dtype=fa.FA_F32) == fa.FA_ERR_UNSUPPORTED
    assert merge(d=96) == fa.FA_ERR_HEADDIM
    assert merge(O=A + 2) == fa.FA_ERR_ALIGN
    assert merge(L=A + 1) == fa.FA_ERR_ALIGN


def test_backward_workspace_size_formula(L):
    def part(n):
        return (n + 255) // 256 * 256
    # fp32 dQ accumulator, then two fp32 values per row of the 128-row padded layout
    assert fa.fa_bwd_workspace_size(2, 3, 300, 64) == part(6 * 300 * 64 * 4) + 2 * part(6 * 384 * 4)
    assert fa.fa_bwd_workspace_size(8, 32, 4096, 128) == part(256 * 4096 * 128 * 4) + 2 * part(256 * 4096 * 4)
    assert fa.fa_bwd_workspace_size(1, 1, 1, 96) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 64, 64) == 0


W = 1 << 24  # placeholder workspace address, 256-byte aligned (dry runs only)


@pytest.mark.parametrize("change,code", [
    ({"Q": 0}, fa.FA_ERR_NULL),
    ({"dO": 0}, fa.FA_ERR_NULL),
    ({"dV": 0}, fa.FA_ERR_NULL),
    ({"dtype": 9}, fa.FA_ERR_DTYPE),
    ({"dtype": fa.FA_F32}, fa.FA_ERR_UNSUPPORTED),
    ({"N": 0}, fa.FA_ERR_SHAPE),
    ({"d": 96}, fa.FA_ERR_HEADDIM),
    ({"scale": float("inf")}, fa.FA_ERR_SCALE),
    ({"dK": A + 8}, fa.FA_ERR_ALIGN),
    ({"LSE": A + 2}, fa.FA_ERR_ALIGN),
    ({"ws": 0}, fa.FA_ERR_WORKSPACE),
    ({"ws": W + 64}, fa.FA_ERR_WORKSPACE),
    ({"ws_bytes": 1024}, fa.FA_ERR_WORKSPACE),
])
def test_backward_argument_errors_return_before_launch(D, change, code):
    a = dict(Q=A, K=A, V=A, O=A, dO=A, LSE=A, dQ=A, dK=A, dV=A, B=1, H=2, N=200, d=64, scale=0.125,
             dtype=fa.FA_BF16, ws=W, ws_bytes=1 << 30)
    a.update(change)
    assert D.fa_bwd(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["LSE"], a["dQ"], a["dK"], a["dV"], a["B"], a["H"],
                     a["N"], a["d"], a["scale"], a["dtype"], a["ws"], a["ws_bytes"], None) == code


def test_d256_split_queries(L):
    """d = 256 splits over 64-key tiles (128-row Q tiles): an explicit count
    needs partial rows for every row."""
    assert fa.fa_fwd_splitkv_workspace_size(1, 8, 16384, 256, 4) == _partials_bytes(4 * 8 * 16384, 256)
    # N = 300 has 5 tiles of 64 keys: a request for 9 ranges gets 5
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 300, 256, 9) == _partials_bytes(5 * 300, 256)
    # the backward at d = 256: fp32 dQ accumulator and two rows of statistics
    assert fa.fa_bwd_workspace_size(1, 8, 1000, 256) == \
        (8 * 1000 * 256 * 4 + 255) // 256 * 256 + 2 * ((8 * 1024 * 4 + 255) // 256 * 256)


def _partials_bytes(rows, d):
    """Workspace of fp32 O partials (256-byte aligned) followed by fp32 LSE partials."""
    return (rows * d * 4 + 255) // 256 * 256 + rows * 4


def _unit_shape(d):
    """(Q rows per work unit, keys per K/V tile) of the 16-bit forward kernels."""
    return (128, 64) if d == 256 else (256, 128)


def _tail_expectation(B, H, N, d, num_sms):
    """The wave-tail plan written out: the full waves of Q blocks run unsplit,
    the units of the last partial wave are split as many ways as fit in one
    wave (at most 16, at most one range per K/V tile), and only their rows
    need partial buffers."""
    qr, kt = _unit_shape(d)
    nqb = -(-N // qr)
    units = B * H * nqb
    full, tail = divmod(units, num_sms)
    tiles = -(-N // kt)
    s = min(num_sms // tail, tiles, 16)
    per = -(-tiles // s)
    s = -(-tiles // per)
    first = full * num_sms
    row0 = (first // nqb) * N + (first % nqb) * qr
    return s, first, _partials_bytes(s * (B * H * N - row0), d)


@pytest.mark.parametrize("B,H,N,d,num_sms", [
    (1, 8, 16000, 128, 152),   # 504 units (N not a multiple of 256): 3 full waves, 48 left split 3 ways
    (1, 8, 16000, 128, 148),   # 60 left, split 2 ways
    (1, 4, 10000, 128, 152),   # 160 units: 1 full wave, 8 left split 16 ways
    (8, 12, 2000, 128, 152),   # 768 units (N not a multiple of 256: no streamed tail): 5 full waves, 8 left
    (1, 4, 16384, 256, 152),   # d = 256: 512 units of 128 rows, 3 full waves, 56 left split 2 ways
])
def test_splitkv_plan_tail_on_the_host(L, B, H, N, d, num_sms):
    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, d, 0, num_sms)
    assert rc == fa.FA_OK
    s, first, ws = _tail_expectation(B, H, N, d, num_sms)
    assert p == {"splits": s, "first_split_unit": first, "launches": 3, "workspace_bytes": ws}


def test_splitkv_plan_uniform_and_unsplit_on_the_host(L):
    # explicit counts split every unit alike: workspace for every row
    rc, p = fa.fa_fwd_splitkv_plan(1, 8, 16384, 128, 3, 152)
    assert rc == fa.FA_OK and p == {"splits": 3, "first_split_unit": 0, "launches": 2,
                                    "workspace_bytes": _partials_bytes(3 * 8 * 16384, 128)}
    assert fa.fa_fwd_splitkv_workspace_size(1, 8, 16384, 128, 3) == p["workspace_bytes"]
    # clamped to whole 128-key tiles: N = 300 has 3
    rc, p = fa.fa_fwd_splitkv_plan(1, 1, 300, 64, 9, 152)
    assert p == {"splits": 3, "first_split_unit": 0, "launches": 2, "workspace_bytes": _partials_bytes(900, 64)}
    # 4096 units on 152 SMs: the last wave is nearly full (144 units), no split pays
    rc, p = fa.fa_fwd_splitkv_plan(8, 32, 4096, 128, 0, 152)
    assert p == {"splits": 1, "first_split_unit": 4096, "launches": 1, "workspace_bytes": 0}
    # a short last wave whose split saves less than the launch boundary costs:
    # d = 256, B=4 H=16 N=4096 (2048 units, 13.5 waves)
    rc, p = fa.fa_fwd_splitkv_plan(4, 16, 4096, 256, 0, 152)
    assert p == {"splits": 1, "first_split_unit": 2048, "launches": 1, "workspace_bytes": 0}
    # d = 256: explicit counts over 64-key tiles
    rc, p = fa.fa_fwd_splitkv_plan(4, 16, 4096, 256, 8, 152)
    assert p == {"splits": 8, "first_split_unit": 0, "launches": 2,
                 "workspace_bytes": _partials_bytes(8 * 64 * 4096, 256)}
    # an explicit count of 1 never splits
    for args in [(2, 2, 1000, 128, 1, 152), (2, 2, 1000, 256, 1, 152)]:
        rc, p = fa.fa_fwd_splitkv_plan(*args)
        units = args[0] * args[1] * -(-args[2] // _unit_shape(args[3])[0])
        assert rc == fa.FA_OK and p == {"splits": 1, "first_split_unit": units, "launches": 1, "workspace_bytes": 0}


def test_splitkv_plan_invariants_over_shapes(L):
    """Over a sweep of shapes and SM counts: three launches exactly when some
    but not all units are split, and the workspace covers exactly the split
    units' rows, one span per key range."""
    for B, H, N in [(1, 1, 64), (1, 2, 1000), (2, 3, 4097), (1, 8, 16384), (3, 5, 777), (16, 16, 512), (1, 1, 65536)]:
        for d in (64, 128, 256):
            qr, kt = _unit_shape(d)
            for num_sms in (1, 7, 132, 148, 152, 1000):
                for ns in (0, 1, 2, 5):
                    rc, p = fa.fa_fwd_splitkv_plan(B, H, N, d, ns, num_sms)
                    assert rc == fa.FA_OK
                    nqb = -(-N // qr)
                    units = B * H * nqb
                    first, s = p["first_split_unit"], p["splits"]
                    rc, sp = fa.fa_fwd_stream_plan(B, H, N, d, num_sms)
                    assert rc == fa.FA_OK
                    if ns == 0 and sp["ctas"] > 0:
                        # the streamed tail (its own tests check the partition)
                        assert d == 128 and N % 256 == 0 and first == sp["unit0"] and p["launches"] == 2
                        assert p["workspace_bytes"] >= 2 * sp["ctas"] * 256 * (4 * d + 4)
                        continue
                    if s == 1:
                        assert first == units and p["launches"] == 1 and p["workspace_bytes"] == 0
                        continue
                    assert 1 < s <= max(ns, 16) and s <= -(-N // kt)
                    assert p["launches"] == (3 if 0 < first < units else 2)
                    assert ns == 0 or first == 0
                    row0 = (first // nqb) * N + (first % nqb) * qr
                    assert p["workspace_bytes"] == _partials_bytes(s * (B * H * N - row0), d)


def test_splitkv_plan_argument_errors(L):
    import ctypes
    assert fa.fa_fwd_splitkv_plan(1, 1, 64, 64, 0, 0)[0] == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_splitkv_plan(0, 1, 64, 64, 0, 152)[0] == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_splitkv_plan(1, 1, 64, 64, -1, 152)[0] == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_splitkv_plan(1, 1, 64, 96, 0, 152)[0] == fa.FA_ERR_HEADDIM
    assert fa.fa_fwd_splitkv_plan(65536, 65536, 64, 64, 0, 152)[0] == fa.FA_ERR_SHAPE
    assert L.fa_fwd_splitkv_plan(1, 1, 64, 64, 0, 152, None, None, None, None) == fa.FA_ERR_NULL
    s = ctypes.c_int()
    assert L.fa_fwd_splitkv_plan(1, 1, 64, 64, 0, 152, ctypes.byref(s), None, None, None) == fa.FA_ERR_NULL
