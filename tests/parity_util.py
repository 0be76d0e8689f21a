"""Comparison of the CUDA path's outputs with the oracle's, with the stated gates.

Gates (max |err| and cosine come from the accuracy thresholds of the dataflow
page's section 4.1; the LSE bound is derived from fp32 accumulation):
  * fp32 inputs:  max |O - O_ref| <= 1e-5;  |dLSE| <= 1e-5 + 1e-6 |LSE_ref|
  * fp16 inputs:  max |O - O_ref| <= 1e-2;  cosine(O, O_ref) >= 0.999
  * bf16 inputs:  the error beyond the rounding of the stored output: for
                  every element, the distance from O_ref to the interval of
                  reals that round to the stored bf16 value is <= 1e-2 (the
                  stored value is the rounding of some number within 1e-2 of
                  the exact result; with sigma-3 inputs |O| reaches ~4.4, where
                  one bf16 half-ulp alone is 0.0156 > 1e-2), cosine >= 0.999;
                  the raw max |err| is reported as well
  * fp16/bf16:    |dLSE| <= 1e-4 * max(1, |LSE_ref|)
"""
import numpy as np
import torch

TOL = {
    "f32": dict(o=1e-5, lse_abs=1e-5, lse_rel=1e-6),
    "f16": dict(o=1e-2, lse_abs=0.0, lse_rel=1e-4, cos=0.999),
    "bf16": dict(o=1e-2, lse_abs=0.0, lse_rel=1e-4, cos=0.999),
}


def dtype_name(t):
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def bf16_rounding_excess(o, o_ref: np.ndarray) -> np.ndarray:
    """Per element, the distance from o_ref to the interval of reals that
    round (to nearest even) to the bf16 value o: 0 when o is the rounding of
    o_ref itself. bf16 keeps 8 significant bits, so a value y with
    2^e <= |y| < 2^(e+1) has neighbours 2^(e-7) away, except 2^(e-8) below
    a power of two; the interval reaches halfway to each neighbour."""
    y = np.asarray(o, dtype=np.float64)
    a = np.abs(y)
    m, e = np.frexp(a)                       # a = m * 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, e - 8)               # 2^(floor(log2 a) - 7)
    away = ulp / 2                           # half-gap away from zero
    toward = np.where(m == 0.5, ulp / 4, ulp / 2)  # half-gap towards zero
    lo = np.where(y >= 0, y - toward, y - away)
    hi = np.where(y >= 0, y + away, y + toward)
    zero = a == 0
    lo = np.where(zero, 0.0, lo)
    hi = np.where(zero, 0.0, hi)
    return np.maximum(0.0, np.maximum(lo - o_ref, o_ref - hi))


def rounding_floor(o_ref: np.ndarray, dtype: str) -> np.ndarray:
    """|round_to_dtype(O_ref) - O_ref|: the error any stored output of that dtype carries."""
    t = torch.from_numpy(o_ref)
    r = t.to({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]).double()
    return (r - t).abs().numpy()


def compare(o, lse, o_ref, lse_ref, dtype: str):
    """Returns a dict of error figures and whether every gate holds."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    err = np.abs(o - o_ref)
    tol = TOL[dtype]
    res = {"max_abs": float(err.max()) if err.size else 0.0}
    if dtype == "bf16":
        res["max_excess"] = float(bf16_rounding_excess(o, o_ref).max()) if err.size else 0.0
        o_ok = res["max_excess"] <= tol["o"]
    else:
        o_ok = res["max_abs"] <= tol["o"]
    lse_err = np.abs(lse - lse_ref)
    lse_bound = np.maximum(tol["lse_abs"] + tol["lse_rel"] * np.abs(lse_ref),
                           tol["lse_rel"] if dtype != "f32" else 0.0)
    res["lse_max_abs"] = float(lse_err.max()) if lse_err.size else 0.0
    lse_ok = bool(np.all(lse_err <= lse_bound))
    ok = o_ok and lse_ok and np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    if "cos" in tol:
        a, b = o.reshape(-1), o_ref.reshape(-1)
        res["cos"] = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
        ok = ok and res["cos"] >= tol["cos"]
    res["ok"] = bool(ok)
    return res
