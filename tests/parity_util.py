"""Comparison of the CUDA path's outputs with the oracle's, with the stated gates.

Gates (max |err| and cosine come from the accuracy thresholds of the dataflow
page's section 4.1; the LSE bound is derived from fp32 accumulation):
  * fp32 inputs:  max |O - O_ref| <= 1e-5;  |dLSE| <= 1e-5 + 1e-6 |LSE_ref|
  * fp16 inputs:  max |O - O_ref| <= 1e-2;  cosine(O, O_ref) >= 0.999
  * bf16 inputs:  max over elements of (|O - O_ref| - |rn_bf16(O_ref) - O_ref|) <= 1e-2
                  (the error beyond the unavoidable rounding of the stored bf16
                  output; with sigma-3 inputs |O| reaches ~4.4 where one bf16
                  half-ulp alone is 0.0156), cosine >= 0.999; the raw max |err|
                  is reported as well
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
        excess = err - rounding_floor(o_ref, dtype)
        res["max_excess"] = float(excess.max()) if err.size else 0.0
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
