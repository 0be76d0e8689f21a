"""Benchmark: attention forward TFLOP/s (4*B*H*N^2*d) on GB300, one JSON line.

A step is one forward pass over the whole workload (one kernel launch).
Default workload: B=8, H=32, N=4096, d=128, bf16, Q and K ~ N(0, 3^2), V ~ N(0, 1)
(the largest measured workload; the throughput target applies to N >= 4096, d=128).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

N > 1 runs one process per GPU under torch.distributed.run: every rank runs
the full per-GPU workload (independent (batch, head) problems, no collective on
the data path: weak scaling); the time is the max over ranks.

The `reference` arm times the CPU fp64 oracle (a deliberately slow program) on
a bounded sample of the same workload; it is a baseline, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "b8h32n4096d128_bf16_qk3"
FALLBACK_TFLOPS = 1900.0  # bf16 dense burst measured once on a GB300 (used only if no measured file)
FALLBACK_SUSTAINED_TFLOPS = 1700.0  # the same measurement held for seconds under the power cap
DATASHEET_TFLOPS = 2250.0  # GB300 dense bf16/fp16 tensor peak per GPU, nominal (without 2:4 sparsity)
COMMON_SOURCES = ["exact_attention_87_gb300/csrc/sm103_ptx.cuh", "exact_attention_87_gb300/csrc/fa_device_common.cuh",
                  "exact_attention_87_gb300/csrc/fa_internal.h"]
# The source files of the kernel each timed path spends its time in.
KERNEL_SOURCES = {
    "fwd": ["exact_attention_87_gb300/csrc/fa_fwd_f16.cu", "exact_attention_87_gb300/csrc/fa_fwd_order.cuh"]
    + COMMON_SOURCES,
    "fwd_d256": ["exact_attention_87_gb300/csrc/fa_fwd_d256.cu", "exact_attention_87_gb300/csrc/fa_fwd_order.cuh"]
    + COMMON_SOURCES,
    "bwd": ["exact_attention_87_gb300/csrc/fa_bwd_f16.cu", "exact_attention_87_gb300/csrc/fa_bwd_order.cuh"]
    + COMMON_SOURCES,
    "bwd_d256": ["exact_attention_87_gb300/csrc/fa_bwd_f16.cu", "exact_attention_87_gb300/csrc/fa_bwd_d256.cu",
                 "exact_attention_87_gb300/csrc/fa_bwd_order.cuh"] + COMMON_SOURCES,
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)", m
    except Exception:
        return FALLBACK_TFLOPS, "fallback", {}


def sustained_peak(m: dict):
    """The bf16 dense rate held for seconds under the power cap, and its source."""
    try:
        return float(m["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json bf16_tflops_sustained)"
    except Exception:
        return FALLBACK_SUSTAINED_TFLOPS, "fallback"


def sustained_leg(step, flops_per_step: float, stream, dev, barrier, seconds: float, ms_hint: float) -> dict:
    """The same step back to back for about `seconds` (one event pair around
    all of them), with the SM clock sampled throughout: how the kernel holds
    up once the GPU settles at its power cap."""
    import torch
    n = max(10, int(seconds * 1e3 / max(ms_hint, 1e-3)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    with sampler:
        barrier()
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        barrier()
    ms = e0.elapsed_time(e1) / n
    value = flops_per_step / (ms * 1e-3) / 1e12
    peak, src = sustained_peak(peaks()[2])
    return {"seconds": round(ms * n / 1e3, 3), "steps": n, "value": round(value, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "peak": peak, "peak_source": src, "frac": round(value / peak, 4),
            "clocks": sampler.summary()}


def code_of(text: str) -> str:
    """A source file's code without its comments and blank lines: the traffic
    recorded for a kernel stays valid across edits of its comments only."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_hash(kind: str = "fwd") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kind: str = "fwd"):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        ent = rec.get(workload if kind == "fwd" else f"{workload}:{kind}")
        if ent and ent.get("kernel_hash") == kernel_hash(kind):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable: nvidia-smi gave no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world_size: int, flops_per_rank: float, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s under weak scaling: every rank does the full per-GPU
    workload each step; the step takes as long as the slowest rank."""
    return world_size * flops_per_rank / (ms_per_step_max * 1e-3) / 1e12


L2_BYTES = 129 * 10**6  # GB300 L2
FLUSH_BYTES = 256 * 2**20  # more than L2: overwriting it evicts every line


def l2_policy(input_bytes: int) -> tuple[int, str]:
    """Bytes to overwrite before every timed step (0: none) and the note for `config`."""
    if input_bytes > L2_BYTES:
        return 0, "inputs larger than L2 (no flush)"
    return FLUSH_BYTES, "L2 flushed before every timed step (256 MiB overwritten outside the timed events)"


def timed_steps(step, steps: int, stream, dev, barrier, flush_bytes: int):
    """Time `steps` calls of `step` with CUDA events on `stream`.

    Returns (total ms, per-step ms). Without a flush the total is one event
    pair around `steps` back-to-back steps, and the per-step times come from a
    second pass of `steps` steps with an event pair around each (so the events
    do not perturb the total). With a flush, a buffer of `flush_bytes` is
    overwritten before each step, outside that step's events, and the total
    is the sum of the per-step times of that one pass."""
    import torch

    def per_step_pass(flush):
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier()
        for i, (a, b) in enumerate(pairs):
            if flush is not None:
                flush.fill_(i & 0xFF)
            a.record(stream)
            step()
            b.record(stream)
        barrier()
        return [a.elapsed_time(b) for a, b in pairs]

    if flush_bytes:
        per = per_step_pass(torch.empty(flush_bytes, dtype=torch.uint8, device=dev))
        return sum(per), per
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    total = e0.elapsed_time(e1)
    return total, per_step_pass(None)


def e2e_pipelined(stream, barrier, n_steps: int, host_in, dev_in, host_out, dev_out, compute,
                  copy_streams: int = 1) -> float:
    """ms per step of `n_steps` end-to-end steps through the public API, the
    copies of neighbouring steps overlapped with the kernels.

    Two device buffer sets b = i % 2. Step i: its inputs host_in -> dev_in[b]
    spread over `copy_streams` input streams (once step i-2's kernels have
    finished reading set b), compute(b) on `stream` (once those copies have
    landed and step i-2's outputs have been read back), its outputs
    dev_out[b] -> host_out[b] on an output stream. Every step's copies lie
    inside the timed region. (Three input streams measured no faster than one
    on GB300: the host link carries about 210 GB/s host-to-device and 193 GB/s
    device-to-host, 170 GB/s each with both at once, whoever drives it.)"""
    import torch
    s_in = [torch.cuda.Stream(stream.device) for _ in range(copy_streams)]
    s_out = torch.cuda.Stream(stream.device)
    ev_in = [[torch.cuda.Event() for _ in s_in] for _ in range(2)]
    ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(2))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    a0.record(stream)
    for s in s_in + [s_out]:
        s.wait_stream(stream)
    for i in range(n_steps):
        b = i & 1
        for c, s in enumerate(s_in):
            if i >= 2:
                s.wait_event(ev_comp[b])
            with torch.cuda.stream(s):
                for d, h in list(zip(dev_in[b], host_in))[c::copy_streams]:
                    d.copy_(h, non_blocking=True)
            ev_in[b][c].record(s)
            stream.wait_event(ev_in[b][c])
        if i >= 2:
            stream.wait_event(ev_out[b])
        compute(b)
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out[b], dev_out[b]):
                h.copy_(d, non_blocking=True)
        ev_out[b].record(s_out)
    for s in s_in + [s_out]:
        stream.wait_stream(s)
    a1.record(stream)
    barrier()
    return a0.elapsed_time(a1) / n_steps


def step_distribution(per_ms) -> dict:
    """Median, 10th and 90th percentile of the per-step times (ms)."""
    xs = sorted(per_ms)

    def pct(f):
        i = f * (len(xs) - 1)
        lo = int(i)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (i - lo)

    return {"median": round(pct(0.5), 4), "p10": round(pct(0.1), 4), "p90": round(pct(0.9), 4), "n": len(xs)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_oracle_sample(w, q, k, v, seconds: float, max_heads: int | None = None, causal: bool = False):
    """Time the oracle on whole heads of the workload until about `seconds` pass.
    Returns (flops done, wall seconds, threads, description, results) where
    results holds each timed head's (b, h, O_ref, LSE_ref)."""
    import oracle
    threads = oracle.default_threads()
    flops, t_total, heads, results = 0, 0.0, 0, []
    per_head = 4 * w.d * (w.N * (w.N + 1) // 2 if causal else w.N * w.N)
    # heads spread over the batch: every (b, h) in a fixed shuffled order
    order = [(b, h) for b in range(w.B) for h in range(w.H)]
    order = [order[(i * 7919) % len(order)] for i in range(len(order))] if len(order) % 7919 else order
    for (b, h) in order:
        t0 = time.perf_counter()
        if causal:
            o_ref, l_ref = oracle.attn_masked(q[b, h][None, None], k[b, h][None, None], v[b, h][None, None],
                                              causal=True, scale=w.scale, nthreads=threads)
            o_ref, l_ref = o_ref[0, 0], l_ref[0, 0]
        else:
            o_ref, l_ref = oracle.attn(q[b, h], k[b, h], v[b, h], scale=w.scale, nthreads=threads)
        t_total += time.perf_counter() - t0
        results.append((b, h, o_ref, l_ref))
        flops += per_head
        heads += 1
        if t_total >= seconds or (max_heads and heads >= max_heads):
            break
    desc = (f"{heads} of {w.B * w.H} heads (all {w.N} rows each, fp64 three-pass" +
            (", causal)" if causal else ")"))
    return flops, t_total, threads, desc, results


def bf16_rounding_excess(o, o_ref):
    """Distance from o_ref to the interval of reals that round to the bf16
    value o (0 when o is the rounding of o_ref itself)."""
    import numpy as np
    y = np.asarray(o, dtype=np.float64)
    a = np.abs(y)
    m, e = np.frexp(a)
    ulp = np.ldexp(1.0, e - 8)
    away, toward = ulp / 2, np.where(m == 0.5, ulp / 4, ulp / 2)
    lo = np.where(a == 0, 0.0, np.where(y >= 0, y - toward, y - away))
    hi = np.where(a == 0, 0.0, np.where(y >= 0, y + away, y + toward))
    return np.maximum(0.0, np.maximum(lo - o_ref, o_ref - hi))


def parity_figures(o, lse, results, dtype: str) -> dict:
    """The timed output against the oracle on the CPU-baseline leg's heads:
    max |err|, the bf16 error beyond the rounding of the stored output,
    cosine over those heads and the smallest per-head cosine, max |dLSE|, and
    whether the gates hold (fp16: max |err| <= 1e-2; bf16: error beyond the
    rounding <= 1e-2; both: cosine >= 0.999, |dLSE| <= 1e-4 max(1, |LSE|))."""
    import numpy as np
    max_abs = max_ex = lse_max = 0.0
    dot = n1 = n2 = 0.0
    min_cos, lse_ok = 2.0, True
    for b, h, o_ref, l_ref in results:
        ob = o[b, h].float().cpu().double().numpy()
        lb = lse[b, h].cpu().double().numpy()
        max_abs = max(max_abs, float(np.abs(ob - o_ref).max()))
        if dtype == "bf16":
            max_ex = max(max_ex, float(bf16_rounding_excess(ob, o_ref).max()))
        le = np.abs(lb - l_ref)
        lse_max = max(lse_max, float(le.max()))
        lse_ok = lse_ok and bool(np.all(le <= 1e-4 * np.maximum(1.0, np.abs(l_ref))))
        hd, h1, h2 = float((ob * o_ref).sum()), float((ob * ob).sum()), float((o_ref * o_ref).sum())
        min_cos = min(min_cos, hd / (h1 * h2) ** 0.5)
        dot, n1, n2 = dot + hd, n1 + h1, n2 + h2
    cos = dot / (n1 * n2) ** 0.5
    o_metric = max_ex if dtype == "bf16" else max_abs
    res = {"heads": len(results), "max_abs": round(max_abs, 6), "cos": round(cos, 9),
           "min_head_cos": round(min_cos, 9), "lse_max_abs": float(f"{lse_max:.3e}")}
    if dtype == "bf16":
        res["max_excess_over_rounding"] = round(max_ex, 6)
    res["ok"] = bool(o_metric <= 1e-2 and cos >= 0.999 and min_cos >= 0.999 and lse_ok)
    res["checked"] = "the output of the last timed step, every element of the heads the CPU baseline computed"
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle CPU-baseline budget")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the sustained leg (0: skip it)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask (FLOPs counted for the keys each row sees: 4*d*N*(N+1)/2 per head)")
    ap.add_argument("--splits", type=int, default=None,
                    help="forward split-KV ranges (0 = automatic, the default: unsplit unless the cost model finds "
                         "the wave tail worth splitting; 1 = the plain forward pass); causal runs default to 1, "
                         "backward runs are unsplit")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time the backward pass (fa_bwd: dQ, dK, dV; 10*B*H*N^2*d FLOPs) instead")
    ap.add_argument("--shard", default="none", choices=["none", "heads"],
                    help="heads: one problem split across the ranks in contiguous blocks of its B*H (batch, head) "
                         "problems (strong scaling, no collective); none: every rank runs the whole workload "
                         "(weak scaling)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (smaller captures of the same workload for profiling; not a bench line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.which == "bwd" and args.splits not in (None, 1):
        raise SystemExit("--pass bwd does not take --splits")
    if args.splits is None:
        args.splits = 1 if (args.causal or args.which == "bwd") else 0

    import dataclasses
    from workloads import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    if args.batch is not None:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}[B={args.batch}]")
    flops = w.flops if not args.causal else 4 * w.B * w.H * w.d * w.N * (w.N + 1) // 2
    ws, rank, local = dist_env()
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype, "sigma_qk": w.sigma_qk,
           "sigma_v": w.sigma_v, "scale": "1/sqrt(d)", "causal": False,
           "l2": None}
    # Inputs of one step: Q, K, V (forward) or Q, K, V, O, dO (backward).
    es = 4 if w.dtype == "f32" else 2
    args.flush_bytes, cfg["l2"] = l2_policy((5 if args.which == "bwd" else 3) * w.B * w.H * w.N * w.d * es)
    if args.causal:
        cfg["causal"] = True
        cfg["flops"] = "4*d*N*(N+1)/2 per (b, h)"

    if args.impl == "reference":
        return run_reference(args, w, cfg, ws, rank)
    if args.which == "bwd":
        return run_backward(args, w, cfg, ws, rank, local)

    import torch
    import torch.distributed as dist
    import exact_attention_87_gb300 as fa

    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.build()
    fa.lib()

    q, k, v = make_inputs(w)
    job_flops = flops
    if args.shard == "heads":
        # This rank's contiguous block of the B*H problems of the one workload.
        from exact_attention_87_gb300.head_parallel import head_bounds, head_slice
        lo, hi = head_bounds(w.B, w.H, ws, rank)
        if hi <= lo:
            raise SystemExit("--shard heads needs at least one (batch, head) problem per rank")
        q, k, v = (head_slice(t, lo, hi).contiguous() for t in (q, k, v))
        w = dataclasses.replace(w, B=1, H=hi - lo)
        flops = flops * (hi - lo) // (cfg["B"] * cfg["H"])
        cfg["parallelism"] = f"heads: rank r runs problems head_bounds(B, H, {ws}, r) (no collective)"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws_bytes = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.d, args.splits) if args.splits != 1 else 0
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    # The plan the library runs: 1 launch (unsplit), 2 (every unit split, merge) or 3 (split wave tail).
    n_launch = 1
    streamed = False
    if args.splits != 1 and w.dtype != "f32":
        n_launch = fa.fa_fwd_splitkv_launches(w.B, w.H, w.N, w.d, args.splits)
        if n_launch < 1:
            raise RuntimeError(f"fa_fwd_splitkv_launches failed ({n_launch})")
        n_splits = fa.fa_fwd_splitkv_num_splits(w.B, w.H, w.N, w.d) if args.splits == 0 else args.splits
        cfg["num_splits"] = n_splits if n_launch > 1 else 1
        cfg["launches_per_step"] = n_launch
        if n_launch == 3:
            cfg["split_plan"] = "tail: full waves unsplit, the last wave's units split, their rows merged"
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        rc, sp = fa.fa_fwd_stream_plan(w.B, w.H, w.N, w.d, sms)
        if args.splits == 0 and not args.causal and rc == fa.FA_OK and sp["ctas"] > 0:
            cfg["num_splits"] = 1
            cfg["split_plan"] = (f"streamed tail: units 0..{sp['unit0'] - 1} whole on the persistent kernel, "
                                 f"the {sp['tiles']} K/V tiles of the rest cut into {sp['ctas']} ranges "
                                 f"(one per SM), cut units merged (at most {n_splits} pieces)")
            streamed = True

    def step():
        fa.attention(qd, kd, vd, scale=w.scale, out=o, lse=lse, stream=stream, num_splits=args.splits,
                     workspace=workspace, causal=args.causal)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status error after warm-up")

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    with sampler:
        local_total, per_step = timed_steps(step, args.steps, stream, dev, barrier, args.flush_bytes)
    ms_total = max_over_ranks(local_total, dev)
    ms = ms_total / args.steps
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st} after the timed region")
    # weak: every rank ran the whole workload; strong (--shard heads): the
    # ranks shared one workload, the job's FLOPs over the slowest rank's time
    tflops = job_throughput(ws, flops, ms) if args.shard == "none" else job_flops / (ms * 1e-3) / 1e12
    # The timed steps' output, kept for the parity figures (the e2e leg below reuses the buffers).
    o_timed, lse_timed = o.clone(), lse.clone()
    sustained = (sustained_leg(step, flops, stream, dev, barrier, args.sustained_seconds, ms)
                 if args.sustained_seconds > 0 else None)

    # ---- e2e: public API with host buffers, copies inside the timed region ----
    e2e = None
    if not args.no_e2e:
        host_in = [q.pin_memory(), k.pin_memory(), v.pin_memory()]
        dev_in = [[qd, kd, vd], [torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]]
        dev_out = [[o, lse], [torch.empty_like(o), torch.empty_like(lse)]]
        host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out[0]] for _ in range(2)]
        ws2 = [workspace, torch.empty_like(workspace)]

        def compute(b):
            qb, kb, vb = dev_in[b]
            fa.attention(qb, kb, vb, scale=w.scale, out=dev_out[b][0], lse=dev_out[b][1], stream=stream,
                         num_splits=args.splits, workspace=ws2[b], causal=args.causal)

        e2e_pipelined(stream, barrier, 2, host_in, dev_in, host_out, dev_out, compute)  # warm-up
        n_e2e = max(4, min(args.steps, 10))
        e_ms = max_over_ranks(e2e_pipelined(stream, barrier, n_e2e, host_in, dev_in, host_out, dev_out, compute),
                              dev)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        e2e = {"value": round(job_throughput(ws, flops, e_ms), 2), "unit": "TFLOP/s", "ms_per_step": round(e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "path": "pinned host -> cudaMemcpyAsync (input stream) -> fa_fwd -> cudaMemcpyAsync (output stream) "
                       "-> pinned host; step i+1's input copies and step i-1's output copies overlap step i's kernel"}

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peak, peak_src, _ = peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    kind = "fwd_d256" if w.d == 256 else "fwd"
    traffic = recorded_traffic(w.name, kind) if not args.causal and n_launch == 1 else None
    line = {
        "metric": "attention fwd TFLOP/s (4*B*H*N^2*d) and % of GB300 dense BF16 tensor peak",
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "ms_per_step_dist": step_distribution(per_step),
        "higher_is_better": True,
        "scaling": "weak" if args.shard == "none" else "strong",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded, generated on the host)",
        "config": cfg,
        "pct_of_measured_peak": round(100.0 * achieved / peak, 2),
        "pct_of_datasheet_peak": round(100.0 * achieved / DATASHEET_TFLOPS, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "kernel": fwd_kernel_name(w, args.causal, n_launch, streamed),
                     "traffic": traffic, "algorithmic_bytes": w.hbm_bytes},
        "clocks": sampler.summary(),
        "sustained": sustained,
        "gpu_launches": args.steps * n_launch,
        "e2e": e2e,
    }
    if ws == 1 and not args.no_cpu_baseline:
        flops_s, secs, threads, desc, results = run_oracle_sample(w, q, k, v, args.cpu_seconds, causal=args.causal)
        line["cpu_baseline"] = {"value": round(flops_s / secs / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        line["parity"] = parity_figures(o_timed, lse_timed, results, w.dtype)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def fwd_kernel_name(w, causal: bool = False, launches: int = 1, streamed: bool = False) -> str:
    """The forward kernel a workload's step spends its time in: at d = 128 one
    unsplit launch takes the persistent form when N is a multiple of 256
    (512 with the causal mask) and at most 4096, and so does the streamed
    tail; at d = 64 the unmasked ones with the same N do."""
    t = "bf16" if w.dtype == "bf16" else "f16"
    if w.dtype == "f32":
        return f"fa_fwd_f32_kernel<{w.d}>"
    if w.d == 256:
        return f"fa_fwd_d256_kernel<{t}>"
    if w.d == 128 and (streamed or (launches == 1 and w.N % (512 if causal else 256) == 0 and w.N <= 4096)):
        return f"fa_fwd_persist_kernel<{w.d},{t}>"
    if w.d == 64 and not causal and launches == 1 and w.N % 256 == 0 and w.N <= 4096:
        return f"fa_fwd_persist_kernel<{w.d},{t}>"
    return f"fa_fwd_f16_kernel<{w.d},{t}>"


def bwd_config(cfg, causal: bool) -> dict:
    """The `config` of a backward line (both arms)."""
    cfg = dict(cfg)
    cfg["pass"] = "bwd"
    cfg["flops"] = ("10*B*H*d*N*(N+1)/2 (S, dP, dV, dK, dQ over the causal pairs)" if causal
                    else "10*B*H*N^2*d (S, dP, dV, dK, dQ products)")
    return cfg


def run_backward(args, w, cfg, ws, rank, local):
    """Time the backward pass (fa_bwd: row statistics, main pass, dQ rounding) for
    the workload, given the forward pass's O and LSE and a seeded dO."""
    import torch
    import torch.distributed as dist
    import exact_attention_87_gb300 as fa
    from workloads import make_dout, make_inputs

    causal = bool(args.causal)
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.build()
    fa.lib()
    if causal:  # the five products over the (query, key) pairs each row sees
        flops = 10 * w.B * w.H * w.d * w.N * (w.N + 1) // 2
    else:
        flops = 10 * w.B * w.H * w.N * w.N * w.d  # five N x N x d products per (b, h)
    cfg = bwd_config(cfg, causal)
    q, k, v = make_inputs(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    stream = torch.cuda.current_stream(dev)
    o, lse = fa.attention(qd, kd, vd, scale=w.scale, stream=stream, causal=causal)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wsp = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)

    def step():
        fa.attention_backward(qd, kd, vd, o, lse, dod, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=wsp,
                              stream=stream, causal=causal)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status error after warm-up")

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    with sampler:
        local_total, per_step = timed_steps(step, args.steps, stream, dev, barrier, args.flush_bytes)
    ms = max_over_ranks(local_total, dev) / args.steps
    st = fa.fa_get_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st} after the timed region")
    tflops = job_throughput(ws, flops, ms)

    e2e = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (q, k, v)] + [o.cpu().pin_memory(), lse.cpu().pin_memory(),
                                                         do.pin_memory()]
        dev_in = [[qd, kd, vd, torch.empty_like(o), torch.empty_like(lse), dod],
                  [torch.empty_like(t) for t in (qd, kd, vd, o, lse, dod)]]
        dev_out = [[dq, dk, dv], [torch.empty_like(t) for t in (dq, dk, dv)]]
        host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out[0]] for _ in range(2)]
        wsp2 = [wsp, torch.empty_like(wsp)]

        def compute(b):
            qb, kb, vb, ob, lb, gb = dev_in[b]
            fa.attention_backward(qb, kb, vb, ob, lb, gb, scale=w.scale, dq=dev_out[b][0], dk=dev_out[b][1],
                                  dv=dev_out[b][2], workspace=wsp2[b], stream=stream, causal=causal)

        e2e_pipelined(stream, barrier, 2, host_in, dev_in, host_out, dev_out, compute)  # warm-up
        n_e2e = max(4, min(args.steps, 10))
        e_ms = max_over_ranks(e2e_pipelined(stream, barrier, n_e2e, host_in, dev_in, host_out, dev_out, compute),
                              dev)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        e2e = {"value": round(job_throughput(ws, flops, e_ms), 2), "unit": "TFLOP/s", "ms_per_step": round(e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "path": "pinned host -> cudaMemcpyAsync (input stream) -> " + ("fa_bwd_ex" if causal else "fa_bwd") +
                       " -> cudaMemcpyAsync (output stream) -> pinned host; step i+1's input copies and step "
                       "i-1's output copies overlap step i's kernels"}

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    peak, peak_src, _ = peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    es = 2
    line = {
        "metric": ("attention bwd TFLOP/s (" + ("causal, 10*B*H*d*N*(N+1)/2" if causal else "10*B*H*N^2*d") +
                   ") and % of GB300 dense BF16 tensor peak"),
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "ms_per_step_dist": step_distribution(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded, generated on the host)", "config": cfg,
        "pct_of_measured_peak": round(100.0 * achieved / peak, 2),
        "pct_of_datasheet_peak": round(100.0 * achieved / DATASHEET_TFLOPS, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "kernel": ("whole step: fa_bwd_pre + fa_bwd_dv256 + fa_bwd_dkdq256 + fa_bwd_post" if w.d == 256
                                else "whole step: fa_bwd_pre + fa_bwd_main + fa_bwd_post"),
                     "traffic": None if causal else recorded_traffic(w.name, "bwd_d256" if w.d == 256 else "bwd"),
                     "algorithmic_bytes": 8 * w.B * w.H * w.N * w.d * es + 4 * w.B * w.H * w.N},
        "clocks": sampler.summary(),
        "gpu_launches": (4 if w.d == 256 else 3) * args.steps,
        "e2e": e2e,
    }
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        n = min(w.N, 768)
        threads = oracle.default_threads()
        secs, heads = 0.0, 0
        while secs < args.cpu_seconds and heads < w.B * w.H:
            b, h = divmod(heads, w.H)
            sl = (b, h, slice(0, n))
            qs, ks, vs = (t[sl].unsqueeze(0).unsqueeze(0) for t in (q, k, v))
            dos = do[sl].unsqueeze(0).unsqueeze(0)
            oh, lh = oracle.attn_masked(qs, ks, vs, causal=causal, scale=w.scale, nthreads=threads)
            t0 = time.perf_counter()
            oracle.attn_bwd(qs, ks, vs, oh, dos, lh, scale=w.scale, nthreads=threads, causal=causal)
            secs += time.perf_counter() - t0
            heads += 1
        per_head = 10 * w.d * (n * (n + 1) // 2 if causal else n * n)
        line["cpu_baseline"] = {"value": round(heads * per_head / secs / 1e12, 6), "unit": "TFLOP/s",
                                "cores": 1, "kind": "oracle", "seconds": round(secs, 2),
                                "sample": f"{heads} heads truncated to their first {n} queries and keys "
                                          "(fp64 backward timed; its O, LSE from the forward oracle, untimed; "
                                          "one head runs on one thread)"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args, w, cfg, ws, rank):
    """The oracle, as it stands, on host cores: each step is a bounded sample of the workload
    (forward: query rows of one head against all its keys; backward: one head truncated to its
    first n tokens, the oracle backward timed)."""
    if rank != 0:
        return
    from workloads import make_dout, make_inputs
    import oracle
    q, k, v = make_inputs(w)
    threads = oracle.default_threads()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    causal = bool(args.causal)
    if args.which == "bwd":
        do = make_dout(w.B, w.H, w.N, w.d, w.dtype, seed=0, wid=w.wid)
        n = min(w.N, 512)

        def sl(t, b, h):
            return t[b, h, :n].unsqueeze(0).unsqueeze(0)

        def step(i):
            b, h = heads[i % len(heads)]
            qs, ks, vs, ds = (sl(t, b, h) for t in (q, k, v, do))
            o, lse = oracle.attn_masked(qs, ks, vs, causal=causal, scale=w.scale, nthreads=threads)
            t0 = time.perf_counter()
            oracle.attn_bwd(qs, ks, vs, o, ds, lse, scale=w.scale, nthreads=threads, causal=causal)
            return time.perf_counter() - t0

        flops_per_step = 10 * w.d * (n * (n + 1) // 2 if causal else n * n)
        cfg = bwd_config(cfg, causal)
        metric = ("attention bwd TFLOP/s (" + ("causal, 10*B*H*d*N*(N+1)/2" if causal else "10*B*H*N^2*d") +
                  ") and % of GB300 dense BF16 tensor peak")
        desc = f"per step one (b, h) truncated to its first {n} tokens (fp64 backward timed; its O, LSE untimed)"
    else:
        # size one step: whole key sets, about 1.5 s of CPU work each at most, 64 query rows at least
        t0 = time.perf_counter()
        oracle.attn(q[0, 0, :64], k[0, 0], v[0, 0], scale=w.scale, nthreads=threads)
        per_row = (time.perf_counter() - t0) / 64
        rows = int(max(64, min(w.N, 1.5 / max(per_row, 1e-9))))

        def step(i):
            b, h = heads[i % len(heads)]
            t0 = time.perf_counter()
            if causal:
                # the first `rows` queries see keys 0..row: the causal rows of the head
                oracle.attn_masked(q[b, h, :rows].unsqueeze(0).unsqueeze(0), k[b, h, :rows].unsqueeze(0).unsqueeze(0),
                                   v[b, h, :rows].unsqueeze(0).unsqueeze(0), causal=True, scale=w.scale,
                                   nthreads=threads)
            else:
                oracle.attn(q[b, h, :rows], k[b, h], v[b, h], scale=w.scale, nthreads=threads)
            return time.perf_counter() - t0

        flops_per_step = 4 * w.d * (rows * (rows + 1) // 2 if causal else rows * w.N)
        metric = "attention fwd TFLOP/s (4*B*H*N^2*d) and % of GB300 dense BF16 tensor peak"
        desc = (f"per step the first {rows} query rows of one (b, h) against " +
                ("the keys each sees (causal)" if causal else f"all {w.N} keys") + " (fp64 three-pass)")

    for i in range(args.warmup):
        step(i)
    secs = sum(step(args.warmup + i) for i in range(args.steps))
    value = args.steps * flops_per_step / secs / 1e12
    ms = secs / args.steps * 1e3
    line = {
        "metric": metric,
        "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)", "config": cfg,
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
