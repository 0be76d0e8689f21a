"""GB300 (sm_103a) FlashAttention forward and backward passes.

Python binding of the C ABI in ``include/fa.h``: argument marshalling only.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU fallback. If the compiled library is missing, every call raises.

    import exact_attention_87_gb300 as fa
    O, LSE = fa.attention(q, k, v)          # q, k, v: [B, H, N, d] CUDA tensors
    dQ, dK, dV = fa.attention_backward(q, k, v, O, LSE, dO)

``fa_fwd`` / ``fa_get_device_status`` / ``fa_strerror`` / ``fa_abi_version``
are the C entry points under the same names (pointers as Python ints).
"""
from __future__ import annotations

import ctypes
import math
import os

from ._build import LIB_PATH, build

FA_F32, FA_F16, FA_BF16 = 0, 1, 2
FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_DTYPE", 3: "FA_ERR_SHAPE", 4: "FA_ERR_HEADDIM",
    5: "FA_ERR_ALIGN", 6: "FA_ERR_CUDA", 7: "FA_ERR_DEVICE_TIMEOUT", 8: "FA_ERR_ARCH", 9: "FA_ERR_SCALE",
    10: "FA_ERR_WORKSPACE", 11: "FA_ERR_SCRATCH_LIMIT", 12: "FA_ERR_UNSUPPORTED", 13: "FA_ERR_DEVICE_SMEM",
}
for _code, _name in STATUS_NAMES.items():
    globals()[_name] = _code


class FAError(RuntimeError):
    def __init__(self, code: int, where: str = "fa_fwd"):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({fa_strerror(code)})")


_lib = None


def lib(path: str | None = None):
    """The loaded C library. Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with exact_attention_87_gb300._build.build() "
            "(nvcc for sm_103a); this package has no CPU fallback")
    L = ctypes.CDLL(path)
    vp, i, f, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    L.fa_fwd.restype = i
    L.fa_get_device_status.argtypes = [vp]
    L.fa_get_device_status.restype = i
    L.fa_strerror.argtypes = [i]
    L.fa_strerror.restype = ctypes.c_char_p
    L.fa_abi_version.argtypes = []
    L.fa_abi_version.restype = i
    L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, u64, vp]
    L.fa_fwd_splitkv.restype = i
    L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, vp]
    L.fa_fwd_ex.restype = i
    L.fa_fwd_splitkv_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, i, vp, u64, vp]
    L.fa_fwd_splitkv_ex.restype = i
    L.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    L.fa_fwd_splitkv_noalloc.restype = i
    L.fa_fwd_splitkv_num_splits.argtypes = [i, i, i, i]
    L.fa_fwd_splitkv_num_splits.restype = i
    L.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_fwd_splitkv_workspace_size.restype = u64
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, u64, vp]
    L.fa_bwd.restype = i
    L.fa_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, vp, u64, vp]
    L.fa_bwd_ex.restype = i
    L.fa_fwd_splitkv_launches.argtypes = [i, i, i, i, i]
    L.fa_fwd_splitkv_launches.restype = i
    L.fa_fwd_splitkv_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_ulonglong)]
    L.fa_fwd_splitkv_plan.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    L.fa_fwd_stream_plan.argtypes = [i, i, i, i, i, ip, ip, ip]
    L.fa_fwd_stream_plan.restype = i
    L.fa_fwd_partial.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.fa_fwd_partial.restype = i
    L.fa_merge.argtypes = [vp, vp, i, vp, vp, i, i, i, i, i, vp]
    L.fa_merge.restype = i
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    L.fa_bwd_workspace_size.restype = u64
    if path == LIB_PATH:
        _lib = L
    return L


# ---- C entry points, same names ----

def fa_fwd(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream=None) -> int:
    return lib().fa_fwd(Q, K, V, O, LSE, B, H, N, d, scale, dtype, stream)


def fa_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, dtype, causal, seqlens_k, stream=None) -> int:
    return lib().fa_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, dtype, causal, seqlens_k, stream)


def fa_fwd_splitkv(Q, K, V, O, LSE, B, H, N, d, scale, dtype, num_splits, workspace, workspace_bytes,
                   stream=None) -> int:
    return lib().fa_fwd_splitkv(Q, K, V, O, LSE, B, H, N, d, scale, dtype, num_splits, workspace,
                                workspace_bytes, stream)


def fa_fwd_splitkv_ex(Q, K, V, O, LSE, B, H, N, d, scale, dtype, causal, seqlens_k, num_splits, workspace,
                      workspace_bytes, stream=None) -> int:
    return lib().fa_fwd_splitkv_ex(Q, K, V, O, LSE, B, H, N, d, scale, dtype, causal, seqlens_k, num_splits,
                                   workspace, workspace_bytes, stream)


def fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, B, H, N, d, scale, dtype, num_splits, stream=None) -> int:
    """fa_fwd_splitkv using the library's built-in 32 MiB scratch: for callers
    that may not allocate device memory (see include/fa.h)."""
    return lib().fa_fwd_splitkv_noalloc(Q, K, V, O, LSE, B, H, N, d, scale, dtype, num_splits, stream)


def fa_fwd_splitkv_num_splits(B, H, N, d) -> int:
    return lib().fa_fwd_splitkv_num_splits(B, H, N, d)


def fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits) -> int:
    return lib().fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, workspace, workspace_bytes,
           stream=None) -> int:
    return lib().fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, workspace, workspace_bytes,
                        stream)


def fa_fwd_splitkv_launches(B, H, N, d, num_splits) -> int:
    return lib().fa_fwd_splitkv_launches(B, H, N, d, num_splits)


def fa_fwd_splitkv_plan(B, H, N, d, num_splits, num_sms) -> tuple[int, dict | None]:
    """(status, plan) with plan = {splits, first_split_unit, launches,
    workspace_bytes} for a device with num_sms SMs (host arithmetic only)."""
    s, f, n, w = ctypes.c_int(), ctypes.c_longlong(), ctypes.c_int(), ctypes.c_ulonglong()
    rc = lib().fa_fwd_splitkv_plan(B, H, N, d, num_splits, num_sms, ctypes.byref(s), ctypes.byref(f),
                                   ctypes.byref(n), ctypes.byref(w))
    if rc != FA_OK:
        return rc, None
    return rc, {"splits": s.value, "first_split_unit": f.value, "launches": n.value, "workspace_bytes": w.value}


def fa_fwd_stream_plan(B, H, N, d, num_sms) -> tuple[int, dict | None]:
    """(status, plan) with plan = {unit0, tiles, ctas}: the streamed tail of the
    automatic plan for unmasked 16-bit inputs on a device with num_sms SMs
    (ctas = 0: not streamed; host arithmetic only)."""
    u, t, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib().fa_fwd_stream_plan(B, H, N, d, num_sms, ctypes.byref(u), ctypes.byref(t), ctypes.byref(c))
    if rc != FA_OK:
        return rc, None
    return rc, {"unit0": u.value, "tiles": t.value, "ctas": c.value}


def fa_fwd_partial(Q, K, V, O_part, LSE_part, B, H, Nq, Nk, d, scale, dtype, stream=None) -> int:
    return lib().fa_fwd_partial(Q, K, V, O_part, LSE_part, B, H, Nq, Nk, d, scale, dtype, stream)


def fa_merge(O_parts, LSE_parts, num_parts, O, LSE, B, H, N, d, dtype, stream=None) -> int:
    return lib().fa_merge(O_parts, LSE_parts, num_parts, O, LSE, B, H, N, d, dtype, stream)


def fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, causal, seqlens_k, workspace,
              workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, dtype, causal, seqlens_k, workspace,
                           workspace_bytes, stream)


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return lib().fa_bwd_workspace_size(B, H, N, d)


def fa_get_device_status(stream=None) -> int:
    return lib().fa_get_device_status(stream)


def fa_strerror(code: int) -> str:
    try:
        return lib().fa_strerror(code).decode()
    except ImportError:
        return "library not loaded"


def fa_abi_version() -> int:
    return lib().fa_abi_version()


# ---- torch convenience wrapper (memory and streams only) ----

def _dtype_code(t):
    import torch
    codes = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def attention(q, k, v, scale: float | None = None, out=None, lse=None, stream=None, num_splits: int = 1,
              workspace=None, causal: bool = False, seqlens_k=None):
    """O, LSE for q, k, v of shape [B, H, N, d] (contiguous CUDA tensors, same dtype).

    Returns O (same dtype as q) and LSE (fp32 [B, H, N], natural log). ``out`` and
    ``lse`` may be preallocated; ``stream`` defaults to torch's current stream.
    ``num_splits`` != 1 runs the split-KV path (0 = automatic count); its
    workspace is allocated with torch unless a CUDA uint8 tensor is given.
    ``causal`` / ``seqlens_k`` (CUDA int32 tensor [B] of key lengths) select the
    masked pass, unsplit or (``num_splits`` != 1) split.
    """
    import torch
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError(f"q, k, v must share one [B, H, N, d] shape: {q.shape} {k.shape} {v.shape}")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous ([B, H, N, d] row-major)")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(q.device):
        masked = causal or seqlens_k is not None
        kl = None
        if seqlens_k is not None:
            if seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda or seqlens_k.numel() != B:
                raise ValueError("seqlens_k must be a CUDA int32 tensor of B lengths")
            seqlens_k = seqlens_k.contiguous()
            kl = seqlens_k.data_ptr()
        if masked and num_splits == 1:
            rc = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           B, H, N, d, float(scale), _dtype_code(q), int(bool(causal)), kl, stream)
        elif masked:
            need = fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
            rc = fa_fwd_splitkv_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, H, N, d, float(scale), _dtype_code(q), int(bool(causal)), kl, num_splits,
                                   workspace.data_ptr(), workspace.numel(), stream)
        elif num_splits == 1:
            rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, H, N, d, float(scale), _dtype_code(q), stream)
        else:
            need = fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
            rc = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, H, N, d, float(scale), _dtype_code(q), num_splits, workspace.data_ptr(),
                                workspace.numel(), stream)
    if rc != FA_OK:
        raise FAError(rc)
    return out, lse


def _stream_handle(stream, device):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def attention_partial(q, k, v, scale: float | None = None, o_part=None, lse_part=None, stream=None):
    """One part of attention over a split key set (fa_fwd_partial): all queries
    q [B, H, Nq, d] against the keys k, v [B, H, Nk, d] (16-bit, contiguous CUDA
    tensors). Returns this part's normalised O (fp32 [B, H, Nq, d]) and LSE
    (fp32 [B, H, Nq]); ``merge_partials`` combines parts. An empty key set
    (Nk = 0) gives O = 0, LSE = -inf without a launch."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError(f"q [B, H, Nq, d] and k, v [B, H, Nk, d] expected: {q.shape} {k.shape} {v.shape}")
    if not (q.dtype == k.dtype == v.dtype) or not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors of one dtype")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_part = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device) if o_part is None else o_part
    lse_part = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse_part is None else lse_part
    if o_part.shape != (B, H, Nq, d) or o_part.dtype != torch.float32 or not o_part.is_contiguous():
        raise ValueError("o_part must be a contiguous fp32 [B, H, Nq, d] tensor")
    if lse_part.shape != (B, H, Nq) or lse_part.dtype != torch.float32 or not lse_part.is_contiguous():
        raise ValueError("lse_part must be a contiguous fp32 [B, H, Nq] tensor")
    if Nk == 0:
        o_part.zero_()
        lse_part.fill_(float("-inf"))
        return o_part, lse_part
    with torch.cuda.device(q.device):
        rc = fa_fwd_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                            B, H, Nq, Nk, d, float(scale), _dtype_code(q), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_partial")
    return o_part, lse_part


def merge_partials(o_parts, lse_parts, dtype, out=None, lse=None, stream=None):
    """Merge parts over disjoint key sets (fa_merge): o_parts fp32
    [P, B, H, N, d], lse_parts fp32 [P, B, H, N] (contiguous CUDA tensors) ->
    O of ``dtype`` (torch.float16 / torch.bfloat16) [B, H, N, d] and LSE fp32
    [B, H, N]."""
    import torch
    if o_parts.dim() != 5 or lse_parts.shape != o_parts.shape[:4]:
        raise ValueError(f"o_parts [P, B, H, N, d] and lse_parts [P, B, H, N] expected: {o_parts.shape} {lse_parts.shape}")
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("parts must be fp32")
    if not (o_parts.is_cuda and lse_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("parts must be contiguous CUDA tensors")
    P, B, H, N, d = o_parts.shape
    out = torch.empty((B, H, N, d), dtype=dtype, device=o_parts.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device) if lse is None else lse
    if out.shape != (B, H, N, d) or out.dtype != dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, H, N, d] tensor of dtype")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F16 if dtype == torch.float16 else FA_F32
    with torch.cuda.device(o_parts.device):
        rc = fa_merge(o_parts.data_ptr(), lse_parts.data_ptr(), P, out.data_ptr(), lse.data_ptr(), B, H, N, d, code,
                      _stream_handle(stream, o_parts.device))
    if rc != FA_OK:
        raise FAError(rc, "fa_merge")
    return out, lse


def attention_backward(q, k, v, o, lse, do, scale: float | None = None, dq=None, dk=None, dv=None, workspace=None,
                       stream=None, causal: bool = False, seqlens_k=None):
    """dQ, dK, dV for the forward pass O, LSE = attention(q, k, v, scale) and the
    output gradient do (all [B, H, N, d] contiguous CUDA tensors of one 16-bit
    dtype; lse fp32 [B, H, N]). ``dq``/``dk``/``dv`` may be preallocated; the
    workspace (fa_bwd_workspace_size bytes) is allocated with torch unless a
    CUDA uint8 tensor is given; ``stream`` defaults to torch's current stream.
    ``causal`` / ``seqlens_k`` (CUDA int32 tensor [B]) are the masks the
    forward pass was run with (fa_bwd_ex).
    """
    import torch
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype: {tuple(t.shape)} {t.dtype}")
    if q.dim() != 4:
        raise ValueError(f"q must be [B, H, N, d]: {tuple(q.shape)}")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be an fp32 [B, H, N] tensor")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor like q")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    with torch.cuda.device(q.device):
        need = fa_bwd_workspace_size(B, H, N, d)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        if causal or seqlens_k is not None:
            kl = None
            if seqlens_k is not None:
                if seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda or seqlens_k.numel() != B:
                    raise ValueError("seqlens_k must be a CUDA int32 tensor of B lengths")
                seqlens_k = seqlens_k.contiguous()
                kl = seqlens_k.data_ptr()
            rc = fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), _dtype_code(q),
                           int(bool(causal)), kl, workspace.data_ptr(), workspace.numel(), stream)
            name = "fa_bwd_ex"
        else:
            rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), _dtype_code(q),
                        workspace.data_ptr(), workspace.numel(), stream)
            name = "fa_bwd"
    if rc != FA_OK:
        raise FAError(rc, name)
    return dq, dk, dv


__all__ = ["attention", "attention_backward", "attention_partial", "merge_partials", "fa_fwd_partial", "fa_merge",
           "fa_fwd_splitkv_launches", "fa_fwd_splitkv_plan", "fa_fwd_stream_plan",
           "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_size", "fa_fwd", "fa_fwd_ex", "fa_fwd_splitkv", "fa_fwd_splitkv_ex", "fa_fwd_splitkv_noalloc", "fa_fwd_splitkv_num_splits",
           "fa_fwd_splitkv_workspace_size",
           "fa_get_device_status", "fa_strerror", "fa_abi_version", "build", "lib",
           "FAError", "FA_F32", "FA_F16", "FA_BF16", "FA_OK"]
