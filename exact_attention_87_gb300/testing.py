"""Binding of the TESTING build (libfa_gb300_testing.so, -DFA_TESTING).

Used by the tests only: per-tile running statistics, pipeline timelines and
fault injection for the bounded barrier waits (see include/fa_testing.h).
"""
from __future__ import annotations

import ctypes
import math

from . import FA_OK, FAError, _dtype_code
from ._build import TESTING_LIB_PATH, build

TRACE_CTAS, TRACE_EVENTS, TRACE_TILES = 8, 32, 64
EVENTS = ["S0_issued", "S1_issued", "PV0_issued", "PV1_issued", "sm0_sfull", "sm0_parrive", "sm1_sfull",
          "sm1_parrive", "K_issued", "V_issued", "mma_kfull", "mma_vfull", "cta",
          "sm0_loaded", "sm0_voted", "sm0_pdone", "sm0_stored", "sm1_loaded", "sm1_voted", "sm1_pdone", "sm1_stored"]
def kv_tile(d: int) -> int:
    """Keys per K/V tile of the 16-bit forward kernel for head dimension d
    (stats_trace has ceil(N / kv_tile(d)) entries per row): 128 for d = 64
    and 128, 64 for d = 256."""
    return 64 if d == 256 else 128
_lib = None


def lib():
    """The testing library, with the product entry points bound as in the
    package plus the testing ones."""
    global _lib
    if _lib is None:
        build(testing=True)
        from . import lib as _product_binding
        L = _product_binding(TESTING_LIB_PATH)
        vp, i, f, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
        L.fa_fwd_debug.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, f, vp]
        L.fa_fwd_debug.restype = i
        L.fa_testing_set_dry_run.argtypes = [i]
        L.fa_testing_set_dry_run.restype = None
        L.fa_fwd_testing.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, vp, ll]
        L.fa_fwd_testing.restype = i
        u64 = ctypes.c_ulonglong
        L.fa_bwd_testing.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, u64, vp, i, vp, ll]
        L.fa_bwd_testing.restype = i
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_size.restype = u64
        L.fa_get_device_status.argtypes = [vp]
        L.fa_get_device_status.restype = i
        L.fa_testing_last_timeout_where.restype = ctypes.c_uint
        L.fa_testing_stream_piece.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
        L.fa_testing_stream_piece.restype = i
        L.fa_testing_bwd_tile.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
        L.fa_testing_bwd_tile.restype = i
        L.fa_testing_fwd_unit.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
        L.fa_testing_fwd_unit.restype = i
        _lib = L
    return _lib


def attention(q, k, v, scale=None, inject=0, stats=False, timeline=False, wait_limit_cycles=0, check=True):
    """Like exact_attention_87_gb300.attention, through fa_fwd_testing.

    Returns (O, LSE, stats_trace or None, timeline or None).
    """
    import torch
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    nkv = (N + kv_tile(d) - 1) // kv_tile(d)
    st = torch.zeros((B, H, N, nkv, 2), dtype=torch.float32, device=q.device) if stats else None
    tl = torch.zeros((TRACE_CTAS, TRACE_EVENTS, TRACE_TILES), dtype=torch.int64, device=q.device) if timeline else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib().fa_fwd_testing(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
                              float(scale), _dtype_code(q), stream, int(inject),
                              st.data_ptr() if st is not None else None,
                              tl.data_ptr() if tl is not None else None, int(wait_limit_cycles))
    if check and rc != FA_OK:
        raise FAError(rc, "fa_fwd_testing")
    return out, lse, st, tl


def attention_debug(q, k, v, scale=None, out_f32=False, tau=-1.0, stats=False, check=True):
    """The forward pass through fa_fwd_debug: with out_f32 the output is the
    fp32 O before rounding to the input type; tau is the lazy-rescale
    threshold in log2 units (< 0: the built-in 8; 0: rescale whenever a row's
    max grows). Returns (O, LSE, stats_trace or None)."""
    import torch
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out_f32:
        out16, out32 = None, torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    else:
        out16, out32 = torch.empty_like(q), None
    tile = kv_tile(d)
    st = torch.zeros((B, H, N, (N + tile - 1) // tile, 2), dtype=torch.float32, device=q.device) if stats else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib().fa_fwd_debug(q.data_ptr(), k.data_ptr(), v.data_ptr(), out16.data_ptr() if out16 is not None else None,
                            lse.data_ptr(), B, H, N, d, float(scale), _dtype_code(q), stream,
                            out32.data_ptr() if out32 is not None else None, float(tau),
                            st.data_ptr() if st is not None else None)
    if check and rc != FA_OK:
        raise FAError(rc, "fa_fwd_debug")
    return (out32 if out_f32 else out16), lse, st


class dry_run:
    """Context: the testing library's entry points stop after their argument
    and device checks and enqueue nothing."""

    def __enter__(self):
        lib().fa_testing_set_dry_run(1)
        return lib()

    def __exit__(self, *exc):
        lib().fa_testing_set_dry_run(0)


BWD_EVENTS = ["dV_issued", "dP_issued", "S_next_issued", "dK_issued", "dQ_issued", "sm_S_ready", "sm_P_arrived",
              "sm_dQ_ready", "sm_dQ_reduce_issued", "sm_dP_ready", "sm_dS_arrived", "sm_dS_half_free", "sm_dQ_loaded",
              "cta", "wg1_P_arrived", "wg1_dS_arrived", "dV_ready", "dP_ready", "S_next_ready", "dK_ready", "dQ_ready",
              "Q_load_issued", "dO_load_issued"]


def attention_backward(q, k, v, o, lse, do, scale=None, inject=0, timeline=False, wait_limit_cycles=0, check=True):
    """Like exact_attention_87_gb300.attention_backward, through fa_bwd_testing.

    Returns (dQ, dK, dV, timeline or None).
    """
    import torch
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(lib().fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    tl = torch.zeros((TRACE_CTAS, TRACE_EVENTS, TRACE_TILES), dtype=torch.int64, device=q.device) if timeline else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib().fa_bwd_testing(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), _dtype_code(q),
                              ws.data_ptr(), ws.numel(), stream, int(inject),
                              tl.data_ptr() if tl is not None else None, int(wait_limit_cycles))
    if check and rc != FA_OK:
        raise FAError(rc, "fa_bwd_testing")
    return dq, dk, dv, tl


def device_status(stream=None) -> int:
    return lib().fa_get_device_status(stream)


def last_timeout_where() -> int:
    return lib().fa_testing_last_timeout_where()


def bwd_tile(B: int, H: int, N: int, d: int, causal: bool, cta: int):
    """fa_testing_bwd_tile: (rc, (b*h, key tile)) of backward CTA `cta`."""
    out = (ctypes.c_int * 2)()
    rc = lib().fa_testing_bwd_tile(B, H, N, d, int(causal), cta, out)
    return rc, (out[0], out[1])


def fwd_unit(B: int, H: int, N: int, d: int, causal: bool, unit: int, num_sms: int = 0):
    """fa_testing_fwd_unit: (rc, (b*h, Q block)) of forward work unit `unit`."""
    out = (ctypes.c_int * 2)()
    rc = lib().fa_testing_fwd_unit(B, H, N, d, int(causal), num_sms, unit, out)
    return rc, (out[0], out[1])


def stream_piece(tiles: int, ctas: int, n: int, c: int, q: int):
    """fa_testing_stream_piece: (rc, values) with values the 4 outputs (q >= 0:
    unit, first tile, end tile, slot) or the 2 of q = -1 (c_lo, c_hi)."""
    out = (ctypes.c_int * 4)()
    rc = lib().fa_testing_stream_piece(tiles, ctas, n, c, q, out)
    return rc, list(out[:4] if q >= 0 else out[:2])
