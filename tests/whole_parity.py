"""Whole-tensor parity of a full-size workload against the oracle.

The oracle (three-pass fp64 attention) runs once per workload per test
session, batch index by batch index, and its O and LSE are kept for every
comparison that session makes on that workload (the CUDA path in the
benchmark's launch configuration, unsplit, with O written as fp32, with the
eager rescale). A comparison walks the batch the same way and accumulates, over
EVERY element of O and every row's LSE, the figures of the accuracy thresholds
of the dataflow page, section 4.1 (max |err|, cosine over the whole output),
plus the smallest cosine of any single (b, h) head.

Gates (the `gate` argument):
  "f16":   raw max |O - O_ref| <= 1e-2, cosine >= 0.999
  "bf16":  the error beyond the rounding of the stored output <= 1e-2: the
           distance from O_ref to the interval of reals that round to the
           stored bf16 value (parity_util.bf16_rounding_excess), cosine >= 0.999
  "raw":   raw max |O - O_ref| <= 1e-2, cosine >= 0.999 (O written as fp32
           before rounding: the strict form of the bf16 gate)
and, for all three, |dLSE| <= 1e-4 * max(1, |LSE_ref|) and every output finite;
the minimum per-head cosine must also reach 0.999.

Setting the environment variable FA_PARITY_LOG to a file path appends one JSON
line of figures per comparison to that file.
"""
from __future__ import annotations

import json
import os
import time

import numpy as np
import torch

import oracle
from parity_util import bf16_rounding_excess
from workloads import make_inputs

_CACHE: dict = {}


def oracle_full(w, q=None, k=None, v=None):
    """(O_ref [B,H,N,d] fp64, LSE_ref [B,H,N] fp64, seconds) of workload w."""
    if w.name not in _CACHE:
        if q is None:
            q, k, v = make_inputs(w)
        t0 = time.perf_counter()
        o_ref = np.empty((w.B, w.H, w.N, w.d), dtype=np.float64)
        lse_ref = np.empty((w.B, w.H, w.N), dtype=np.float64)
        for b in range(w.B):
            o_ref[b], lse_ref[b] = oracle.attn(q[b], k[b], v[b], scale=w.scale)
        _CACHE[w.name] = (o_ref, lse_ref, time.perf_counter() - t0)
    return _CACHE[w.name]


def compare_whole(o, lse, o_ref, lse_ref, gate: str, label: str = "") -> dict:
    """Every element of o (device or host tensor [B,H,N,d]) and lse ([B,H,N])
    against the oracle's; returns the figures and whether every gate holds."""
    B, H = o.shape[0], o.shape[1]
    max_abs = max_excess = lse_max = 0.0
    dot = n1 = n2 = 0.0
    min_head_cos, worst_head = 2.0, None
    finite = lse_ok = True
    for b in range(B):
        ob = o[b].detach().to("cpu").double().numpy()
        lb = lse[b].detach().to("cpu").double().numpy()
        rb, rl = o_ref[b], lse_ref[b]
        finite = finite and bool(np.isfinite(ob).all()) and bool(np.isfinite(lb).all())
        err = np.abs(ob - rb)
        max_abs = max(max_abs, float(err.max()))
        if gate == "bf16":
            max_excess = max(max_excess, float(bf16_rounding_excess(ob, rb).max()))
        le = np.abs(lb - rl)
        lse_max = max(lse_max, float(le.max()))
        lse_ok = lse_ok and bool(np.all(le <= 1e-4 * np.maximum(1.0, np.abs(rl))))
        hd = np.einsum("hnd,hnd->h", ob, rb)
        h1 = np.einsum("hnd,hnd->h", ob, ob)
        h2 = np.einsum("hnd,hnd->h", rb, rb)
        hc = hd / np.sqrt(h1 * h2 + 1e-300)
        i = int(np.argmin(hc))
        if hc[i] < min_head_cos:
            min_head_cos, worst_head = float(hc[i]), (b, i)
        dot += float(hd.sum())
        n1 += float(h1.sum())
        n2 += float(h2.sum())
    cos = dot / np.sqrt(n1 * n2 + 1e-300)
    o_metric = max_excess if gate == "bf16" else max_abs
    res = {"label": label, "gate": gate, "max_abs": max_abs, "cos": cos, "min_head_cos": min_head_cos,
           "worst_head": worst_head, "lse_max_abs": lse_max, "finite": finite}
    if gate == "bf16":
        res["max_excess"] = max_excess
    res["ok"] = bool(finite and lse_ok and o_metric <= 1e-2 and cos >= 0.999 and min_head_cos >= 0.999)
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(res) + "\n")
    return res
