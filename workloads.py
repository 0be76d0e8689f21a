"""Seeded synthetic inputs for the attention forward pass.

This module only draws and rounds random numbers. It holds none of the
attention arithmetic, so both the CPU oracle (``oracle/``) and the CUDA path
(``exact_attention_87_gb300``) can take their inputs from it without sharing
any computation.

Recipe (the same bytes go to both sides):
  * one numpy PCG64 stream per tensor: ``default_rng([seed, workload_id, t])``
    with t = 0, 1, 2 for Q, K, V and t = 3 for the output gradient dO of the
    backward pass;
  * ``standard_normal`` drawn in float32, multiplied by the tensor's sigma;
  * rounded once to the workload dtype with round-to-nearest-even
    (numpy ``astype`` for fp16, torch CPU ``.to(torch.bfloat16)`` for bf16).

The workloads are the shapes, dtypes and value distributions on which the
method is measured: a tiny fp32 case for single-tile bring-up, a short fp16
case, a mid-size fp16 case (the worked throughput example on the dataflow page,
B=8, H=12, L=2048, d=128), a large bf16 case whose Q and K have sigma 3 so that
row maxima keep jumping between key tiles, a long-sequence bf16 case, and a
head-dimension-256 bf16 case (the MUSA guide's block-size table goes up to
d = 256), and the 4096-token shape at head dimension 64 (bf16 and fp16), where
the softmax is twice the share of the work.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int          # stream id used in the seed sequence
    B: int
    H: int
    N: int
    d: int
    dtype: str        # "f32" | "f16" | "bf16"
    sigma_qk: float = 1.0
    sigma_v: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> int:
        """4*B*H*N^2*d: two N x N x d contractions per (batch, head)."""
        return 4 * self.B * self.H * self.N * self.N * self.d

    @property
    def hbm_bytes(self) -> int:
        """Q, K, V read once, O written once (dtype), LSE written once (fp32)."""
        es = ELEM_BYTES[self.dtype]
        return 4 * self.B * self.H * self.N * self.d * es + 4 * self.B * self.H * self.N


WORKLOADS = {
    w.name: w
    for w in [
        Workload("b1h1n64d64_f32", 1, 1, 1, 64, 64, "f32"),
        Workload("b1h4n512d64_f16", 2, 1, 4, 512, 64, "f16"),
        Workload("b8h12n2048d128_f16", 3, 8, 12, 2048, 128, "f16"),
        Workload("b8h32n4096d128_bf16_qk3", 4, 8, 32, 4096, 128, "bf16", sigma_qk=3.0),
        Workload("b1h8n16384d128_bf16", 5, 1, 8, 16384, 128, "bf16"),
        Workload("b4h16n4096d256_bf16", 6, 4, 16, 4096, 256, "bf16"),
        Workload("b8h32n4096d64_bf16", 7, 8, 32, 4096, 64, "bf16"),
        Workload("b8h32n4096d64_f16", 8, 8, 32, 4096, 64, "f16"),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(x.astype(np.float16)))
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    raise ValueError(dtype)


def draw(shape, dtype: str, sigma: float, seed: int, wid: int, t: int) -> torch.Tensor:
    """One seeded tensor, already rounded to ``dtype`` (CPU, contiguous)."""
    rng = np.random.default_rng([seed, wid, t])
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return _round(x, dtype)


def make_qkv(B, H, N, d, dtype, sigma_qk=1.0, sigma_v=1.0, seed=0, wid=0, Nk=None):
    """Q [B,H,N,d], K and V [B,H,Nk,d] (Nk defaults to N) as CPU tensors."""
    Nk = N if Nk is None else Nk
    q = draw((B, H, N, d), dtype, sigma_qk, seed, wid, 0)
    k = draw((B, H, Nk, d), dtype, sigma_qk, seed, wid, 1)
    v = draw((B, H, Nk, d), dtype, sigma_v, seed, wid, 2)
    return q, k, v


def make_dout(B, H, N, d, dtype, seed=0, wid=0, sigma=1.0):
    """The output gradient dO [B,H,N,d] for the backward pass (stream t = 3)."""
    return draw((B, H, N, d), dtype, sigma, seed, wid, 3)


def make_inputs(w: Workload | str, seed: int = 0):
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.sigma_qk, w.sigma_v, seed, w.wid)


def rising_norm_order(k: torch.Tensor, v: torch.Tensor):
    """Reorder the keys of each (b, h) by increasing L2 norm, V rows jointly.

    A row's running maximum then tends to grow on every key tile, which makes
    the online-softmax rescale fire as often as possible. This only permutes
    the inputs; the exact result is unchanged by a joint K/V permutation.
    """
    norms = k.float().norm(dim=-1)
    idx = norms.argsort(dim=-1)
    g = idx.unsqueeze(-1).expand_as(k)
    return torch.gather(k, 2, g).contiguous(), torch.gather(v, 2, g).contiguous()
