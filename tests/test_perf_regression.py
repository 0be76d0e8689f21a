"""Throughput against the frozen figures (GPU).

The dataflow page's section 4.5 orders the work: make it run, then tune,
then freeze the best configuration as the baseline that later changes are
measured against. tests/perf_baseline.json holds those figures (TFLOP/s of
bench.py lines on GB300, with the command that produced each). This test
times every entry the same way (the benchmark's launch configuration, inputs
resident, CUDA events on the launching stream after warm-up, the best of
three 10-step medians) and fails when one falls more than 5 % below its
frozen figure. A change that makes a kernel faster should update the file.
"""
import json
import os

import pytest
import torch

import exact_attention_87_gb300 as fa
from workloads import WORKLOADS, make_dout, make_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "perf_baseline.json")) as f:
    BASELINE = json.load(f)["entries"]
TOLERANCE = 0.05


def _flops(w, causal, bwd):
    pairs = w.N * (w.N + 1) // 2 if causal else w.N * w.N
    return (10 if bwd else 4) * w.B * w.H * w.d * pairs


def _median_ms(step, n=10):
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    stream = torch.cuda.current_stream()
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in evs)
    return ts[n // 2]


@pytest.mark.parametrize("key", sorted(BASELINE))
def test_throughput_not_below_frozen_figure(key):
    e = BASELINE[key]
    w = WORKLOADS[e["workload"]]
    causal, bwd = e.get("causal", False), e.get("pass", "fwd") == "bwd"
    fa.build()
    q, k, v = (t.cuda() for t in make_inputs(w))
    if bwd:
        o, lse = fa.attention(q, k, v, causal=causal)
        do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid).cuda()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device="cuda")

        def step():
            fa.attention_backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, causal=causal)
    else:
        splits = e.get("splits", 0)
        o, lse = torch.empty_like(q), torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
        need = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.d, splits) if splits != 1 else 0
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")

        def step():
            fa.attention(q, k, v, out=o, lse=lse, num_splits=splits, workspace=ws, causal=causal)
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    best = min(_median_ms(step) for _ in range(3))
    tflops = _flops(w, causal, bwd) / (best * 1e-3) / 1e12
    assert tflops >= (1 - TOLERANCE) * e["tflops"], \
        f"{key}: {tflops:.1f} TFLOP/s < {(1 - TOLERANCE) * e['tflops']:.1f} ({e['tflops']} frozen)"
