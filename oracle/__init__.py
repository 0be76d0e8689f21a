"""CPU fp64 oracle for the attention forward pass (test infrastructure).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The CUDA
library never loads it and shares no code with it.

What it computes, per (batch, head) and query row i (the standard attention
definition and three-pass safe softmax of the MUSA guide's "FlashAttention 优化"
page, sections "计算流程" and "标准 Softmax 回顾"):

    s_ij  = scale * sum_k q_ik k_jk
    m_i   = max_j s_ij
    Z_i   = sum_j exp(s_ij - m_i)
    O_ik  = sum_j exp(s_ij - m_i) / Z_i * v_jk
    LSE_i = m_i + ln Z_i

all in fp64 from the already-rounded inputs (fp16/bf16/fp32 upcast exactly).
``attn_online`` is the tiled recurrence of the same page's "FlashAttention
完整算法" formula, in fp64, with an optional lazy-rescale threshold.
``merge`` combines results computed over disjoint key ranges with the block
merge of the Triton page (section 2.3), for split-KV. ``attn_masked`` is the
definition restricted to the allowed keys (causal, per-batch key lengths).
``attn_bwd`` is the backward pass by recomputation (the MUSA guide's fourth
core principle, the Triton page's sections 2.4 and 4.4): P is rebuilt from Q,
K and the saved LSE, and the chain rule on the definition gives, with
D_i = sum_c dO_ic O_ic,

    dV = P^T dO,   dS_ij = P_ij (dO_i . v_j - D_i),
    dQ = scale dS K,   dK = scale dS^T Q.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "attn_ref.c")
LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(out: str = LIB, mutant: int = 0) -> str:
    """Compile the oracle with gcc -O2 (no fast-math). Returns the .so path."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
    lib.oracle_attn_fp64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, D, I]
    lib.oracle_attn_fp64.restype = I
    lib.oracle_attn_online_fp64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, D, L, D, dp, dp, I]
    lib.oracle_attn_online_fp64.restype = I
    lp = ctypes.POINTER(ctypes.c_long)
    lib.oracle_attn_masked_fp64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, D, I, lp, I]
    lib.oracle_attn_masked_fp64.restype = I
    lib.oracle_attn_bwd_fp64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, L, L, L, D, I]
    lib.oracle_attn_bwd_fp64.restype = I
    lp = ctypes.POINTER(ctypes.c_long)
    lib.oracle_bwd_rows_fp64.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, D, lp, L, dp, lp, L, dp, dp]
    lib.oracle_bwd_rows_fp64.restype = I
    lib.oracle_attn_bwd_masked_fp64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, L, L, L, D, I, lp, L, I]
    lib.oracle_attn_bwd_masked_fp64.restype = I
    lib.oracle_bwd_rows_masked_fp64.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, D, I, lp, L, lp, L, dp, lp, L,
                                                dp, dp]
    lib.oracle_bwd_rows_masked_fp64.restype = I
    lib.oracle_merge_fp64.argtypes = [dp, dp, L, L, L, dp, dp]
    lib.oracle_merge_fp64.restype = I
    lib.oracle_mutant_id.restype = I
    return lib


def load(path: str | None = None):
    """The default oracle library, built on first use if missing or stale."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        _lib = _bind(LIB)
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (any float dtype, upcast is exact)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, v):
    if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    lead = q.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, q.shape[-2], k.shape[-2], q.shape[-1]


def attn(q, k, v, scale: float | None = None, nthreads: int | None = None, lib=None):
    """Three-pass fp64 attention. q [..., Nq, d], k/v [..., Nk, d] -> (O, LSE) fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead, BH, Nq, Nk, d = _shapes(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty(q.shape, dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    lib = lib or load()
    rc = lib.oracle_attn_fp64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, Nq, Nk, d,
                              scale, nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fp64 failed ({rc})")
    return o, lse


def attn_online(q, k, v, block_n: int, tau: float = 0.0, scale: float | None = None,
                trace: bool = False, nthreads: int | None = None, lib=None):
    """Online (tiled) recurrence in fp64. Returns (O, LSE) or (O, LSE, m_trace, l_trace).

    tau is the lazy-rescale threshold in natural-log units (0 = eager).
    Traces are [..., Nq, nblocks]: the running max and denominator after each block.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead, BH, Nq, Nk, d = _shapes(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty(q.shape, dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    nb = (Nk + block_n - 1) // block_n
    tm = tl = None
    null = ctypes.POINTER(ctypes.c_double)()
    if trace:
        tm = np.empty(q.shape[:-1] + (nb,), dtype=np.float64)
        tl = np.empty_like(tm)
    lib = lib or load()
    rc = lib.oracle_attn_online_fp64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, Nq, Nk, d,
                                     scale, block_n, tau, _ptr(tm) if trace else null,
                                     _ptr(tl) if trace else null, nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_online_fp64 failed ({rc})")
    return (o, lse, tm, tl) if trace else (o, lse)


def attn_masked(q, k, v, causal: bool = False, klen=None, scale: float | None = None,
                nthreads: int | None = None, lib=None):
    """Masked three-pass attention. q [B,H,Nq,d], k/v [B,H,Nk,d]; klen: None or B ints.

    Row i of batch b attends to keys j < klen[b] and, if causal, j <= i. A row
    with no allowed key gets O = 0 and LSE = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4:
        raise ValueError("attn_masked wants [B, H, N, d] arrays")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty(q.shape, dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    kl = None
    if klen is not None:
        kl = np.ascontiguousarray(np.asarray(klen, dtype=np.int64).reshape(-1))
        if kl.shape != (B,):
            raise ValueError("klen must hold one length per batch")
    lib = lib or load()
    lp = kl.ctypes.data_as(ctypes.POINTER(ctypes.c_long)) if kl is not None else ctypes.POINTER(ctypes.c_long)()
    rc = lib.oracle_attn_masked_fp64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, scale,
                                     int(bool(causal)), lp, nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_masked_fp64 failed ({rc})")
    return o, lse


def _klen_arg(klen, B):
    """(array kept alive, C pointer) for per-batch key lengths; NULL pointer for None."""
    lp = ctypes.POINTER(ctypes.c_long)
    if klen is None:
        return None, lp()
    kl = np.ascontiguousarray(np.asarray(klen, dtype=np.int64).reshape(-1))
    if kl.shape != (B,):
        raise ValueError("klen must hold one length per batch")
    return kl, kl.ctypes.data_as(lp)


def attn_bwd(q, k, v, o, do, lse, scale: float | None = None, nthreads: int | None = None, lib=None,
             causal: bool = False, klen=None):
    """Backward pass by recomputation: (dQ, dK, dV) fp64 for q, k, v, do [..., N, d], with the
    forward outputs o [..., N, d] and lse [..., N].

    With masks (``causal``; ``klen``: B key lengths, arrays [B, H, N, d]) a
    masked score is -inf, so its P_ij and dS_ij are exactly 0: masked keys get
    zero dK, dV and contribute nothing to dQ; a row with no key (LSE = -inf,
    O = 0) gets dQ = 0."""
    q, k, v, o, do, lse = (_f64(t) for t in (q, k, v, o, do, lse))
    lead, BH, N, Nk, d = _shapes(q, k, v)
    if Nk != N or o.shape != q.shape or do.shape != q.shape or lse.shape != q.shape[:-1]:
        raise ValueError("attn_bwd wants square attention and matching o / do / lse")
    if klen is not None and q.ndim != 4:
        raise ValueError("attn_bwd with klen wants [B, H, N, d] arrays")
    B, H = (q.shape[0], q.shape[1]) if q.ndim == 4 else (BH, 1)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    kl, klp = _klen_arg(klen, B)
    lib = lib or load()
    rc = lib.oracle_attn_bwd_masked_fp64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                         _ptr(dk), _ptr(dv), BH, N, d, scale, int(bool(causal)), klp, H,
                                         nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_masked_fp64 failed ({rc})")
    return dq, dk, dv


def attn_bwd_rows(q, k, v, o, do, lse, dq_rows, dkv_rows, scale: float | None = None, lib=None,
                  causal: bool = False, klen=None):
    """Selected rows of the backward pass: dQ at (b, h, i) in ``dq_rows`` and
    dK, dV at (b, h, j) in ``dkv_rows``; o and lse must be the forward results
    for every row of the heads named. Returns (dq [n_dq, d], dk, dv [n_dkv, d]).
    ``causal`` and ``klen`` are the masks of ``attn_bwd``."""
    q, k, v, o, do, lse = (_f64(t) for t in (q, k, v, o, do, lse))
    B, H, N, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)

    def pairs(rows):
        a = np.array([[b * H + h, i] for b, h, i in rows], dtype=np.int64).reshape(-1, 2)
        return np.ascontiguousarray(a, dtype=ctypes.c_long)

    a_q, a_kv = pairs(dq_rows), pairs(dkv_rows)
    dq = np.empty((len(a_q), d))
    dk, dv = np.empty((len(a_kv), d)), np.empty((len(a_kv), d))
    lp = ctypes.POINTER(ctypes.c_long)
    kl, klp = _klen_arg(klen, B)
    lib = lib or load()
    rc = lib.oracle_bwd_rows_masked_fp64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), B * H, N, d,
                                         scale, int(bool(causal)), klp, H, a_q.ctypes.data_as(lp), len(a_q),
                                         _ptr(dq), a_kv.ctypes.data_as(lp), len(a_kv), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd_rows_masked_fp64 failed ({rc})")
    return dq, dk, dv


def merge(o_parts, lse_parts, lib=None):
    """Merge results over disjoint key ranges (block merge of the Triton page, section 2.3).

    o_parts [P, ..., d] (each part's normalised O), lse_parts [P, ...] -> (O, LSE) fp64.
    """
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    P = o_parts.shape[0]
    if lse_parts.shape != o_parts.shape[:-1]:
        raise ValueError(f"bad shapes {o_parts.shape} {lse_parts.shape}")
    d = o_parts.shape[-1]
    rows = int(np.prod(o_parts.shape[1:-1])) if o_parts.ndim > 2 else 1
    o = np.empty(o_parts.shape[1:], dtype=np.float64)
    lse = np.empty(lse_parts.shape[1:], dtype=np.float64)
    lib = lib or load()
    rc = lib.oracle_merge_fp64(_ptr(o_parts), _ptr(lse_parts), P, rows, d, _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_merge_fp64 failed ({rc})")
    return o, lse


def attn_rows(q, k, v, rows, scale: float | None = None, nthreads: int | None = None):
    """O and LSE for sampled rows only. rows: list of (b, h, i) into q [B,H,N,d].

    Each sampled row is computed by the three-pass definition against all keys
    of its own (b, h); this lets full-size workloads be checked row by row.
    """
    out_o, out_l = [], []
    by_head: dict = {}
    for n, (b, h, i) in enumerate(rows):
        by_head.setdefault((b, h), []).append((n, i))
    res_o = [None] * len(rows)
    res_l = [None] * len(rows)
    for (b, h), items in by_head.items():
        idx = [i for _, i in items]
        qs = q[b, h, idx]
        o, lse = attn(qs, k[b, h], v[b, h], scale=scale, nthreads=nthreads)
        for t, (n, _) in enumerate(items):
            res_o[n] = o[t]
            res_l[n] = lse[t]
    out_o = np.stack(res_o) if rows else np.zeros((0, q.shape[-1]))
    out_l = np.array(res_l, dtype=np.float64)
    return out_o, out_l


if __name__ == "__main__":  # pragma: no cover
    print(build(*sys.argv[1:2]))
