#!/usr/bin/env python
"""Benchmark of the retention hot path on B300; prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timed step: one ret_chunkwise call on the 7B-shape workload (B2 H16 L8192
d_k256 d_v512, chunk 128, bf16, fp32 state_in), inputs resident in HBM.
The decode workload (batch 128, H16, d_k256, d_v512, fp32 state 1.07 GB) is
timed the same way and reported under "decode".  N > 1 runs one independent
replica per GPU (the path has no exchange step) and reports the aggregate.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunkwise retention tokens/s & % bf16 tensor peak; decode state GB/s % HBM"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="msr7b")
    ap.add_argument("--decode-steps", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--backward-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["chunk7b", "chunk_medium", "gemm", "rownorm7b", "block7b", "gn1p3b", "gnbwd1p3b",
                             "pgrad_medium", "bwd7b", "decode"],
                    help="run one case (two warm-up calls, then one call) for an ncu capture and exit")
    return ap.parse_args()


def run_profile_case(case):
    """One call of one case, after two warm-up calls, for ncu (no timing, no
    JSON line).  chunk7b: ret_chunkwise on the 7B-shape workload; chunk_medium:
    the same shape at L = 2048 (134 MB of inputs, above the 126 MB L2);
    gemm: ret_matmul 8192 x 8192 x 4096; rownorm7b: ret_decay_row_norm on a
    7B-shape bf16 output; block7b: ret_msr_block at the 7B shape; gn1p3b:
    ret_chunkwise with GroupNorm at the 1.3B shape; gnbwd1p3b:
    ret_groupnorm_backward at the 1.3B shape; pgrad_medium:
    ret_chunkwise_param_grads on B1 H4 L4096 d_k256 d_v512; bwd7b:
    ret_chunkwise_backward on the 7B-shape workload (state_in and dS_out);
    decode: ret_step on the decode workload (batch 128, fp32 state 1.07 GB)."""
    import torch
    import linear_recurrent_sequence_prologue_b300 as R
    from linear_recurrent_sequence_prologue_b300 import build
    from linear_recurrent_sequence_prologue_b300.inputs import WORKLOADS, make_inputs
    build.build()
    R.load()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(3)
    rn = lambda shape, std: (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)
    w = WORKLOADS["msr7b"]
    if case == "chunk_medium":
        w = w.with_(L=2048)
    inp = make_inputs(w, seed=0)
    if case in ("chunk7b", "chunk_medium"):
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        s_in = inp["state_in"].to(dev)
        fn = lambda: R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=w.chunk, state_in=s_in)
    elif case == "gemm":
        a, wt = rn((8192, 4096), 1.0), rn((4096, 8192), 4096 ** -0.5)
        fn = lambda: R.matmul(a, wt)
    elif case == "rownorm7b":
        o = rn((w.B, w.H, w.L, w.d_v), 1.0)
        fn = lambda: R.decay_row_norm(o, inp["gamma"])
    elif case == "gn1p3b":
        w3 = WORKLOADS["msr1p3b"]
        i3 = make_inputs(w3, seed=0)
        q, k, v = (i3[n].to(dev) for n in ("q", "k", "v"))
        fn = lambda: R.chunkwise(q, k, v, i3["gamma"], i3["theta"], chunk=w3.chunk, gn={"eps": 1e-5},
                                 return_state=False)
    elif case == "gnbwd1p3b":
        w3 = WORKLOADS["msr1p3b"]
        x, dy = rn((w3.B, w3.H, w3.L, w3.d_v), 1.0), rn((w3.B, w3.H, w3.L, w3.d_v), 1.0)
        gw = torch.randn((w3.H, w3.d_v), generator=gen, device=dev)
        fn = lambda: R.groupnorm_backward(x, dy, 1e-5, gw)
    elif case == "pgrad_medium":
        from linear_recurrent_sequence_prologue_b300.inputs import make_grad_inputs
        wm = w.with_(B=1, H=4, L=4096)
        im = make_inputs(wm, seed=0)
        gi = make_grad_inputs(wm, seed=5, d_state_std=1.0)
        q, k, v, s_in = (im[n].to(dev) for n in ("q", "k", "v", "state_in"))
        d_o, dso = gi["d_out"].to(dev), gi["d_state_out"].to(dev)
        out, _ = R.chunkwise(q, k, v, im["gamma"], im["theta"], chunk=128, state_in=s_in)
        grads = R.chunkwise_backward(q, k, v, d_o, im["gamma"], im["theta"], chunk=128, state_in=s_in,
                                     d_state_out=dso)
        fn = lambda: R.param_grads(q, k, v, d_o, out, *grads[:3], im["gamma"], im["theta"], state_in=s_in,
                                   d_state_out=dso)
    elif case == "decode":
        from linear_recurrent_sequence_prologue_b300.inputs import make_decode_inputs
        dw = WORKLOADS["decode"]
        dinp = make_decode_inputs(dw, seed=0, steps=1, device="cuda:0")
        fn = lambda: R.step(dinp["q"][0], dinp["k"][0], dinp["v"][0], dinp["gamma"], dinp["theta"], 0,
                            dinp["state"])
    elif case == "bwd7b":
        from linear_recurrent_sequence_prologue_b300.inputs import make_grad_inputs
        im = make_inputs(w, seed=0)
        gi = make_grad_inputs(w, seed=5, d_state_std=1.0)
        q, k, v, s_in = (im[n].to(dev) for n in ("q", "k", "v", "state_in"))
        d_o, dso = gi["d_out"].to(dev), gi["d_state_out"].to(dev)
        fn = lambda: R.chunkwise_backward(q, k, v, d_o, im["gamma"], im["theta"], chunk=128, state_in=s_in,
                                          d_state_out=dso)
    else:
        D = w.H * w.d_k
        x = rn((w.B, w.L, D), 1.0)
        ws = [rn((D, w.H, w.d_k), D ** -0.5), rn((D, w.H, w.d_k), D ** -0.5), rn((D, w.H, w.d_v), D ** -0.5),
              rn((D, w.H, w.d_v), D ** -0.5), rn((w.H, w.d_v, D), (w.H * w.d_v) ** -0.5)]
        fn = lambda: R.msr_block(x, *ws, inp["gamma"], inp["theta"])
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    assert R.sync_status() == R.RET_OK
    return 0


# --------------------------------------------------------------------------
# Algorithmic work and bytes of one call, as the chunkwise form states them
# --------------------------------------------------------------------------
def chunk_flops(w):
    """2b·d_k + 2b·d_v + 4·d_k·d_v flop per token per head (QKᵀ, PV, Q·S, KᵀV)."""
    b = w.chunk
    return w.B * w.H * w.L * (2 * b * w.d_k + 2 * b * w.d_v + 4 * w.d_k * w.d_v)


def chunk_bytes(w):
    """Read Q, K, V once, write O once (bf16), read state_in and write state_out (fp32)."""
    return w.B * w.H * w.L * (2 * w.d_k + 2 * w.d_v) * 2 + 2 * w.B * w.H * w.d_k * w.d_v * 4


def decode_bytes(w):
    """Read and write the fp32 state once, plus q, k, v in and o out (bf16)."""
    return 2 * w.B * w.H * w.d_k * w.d_v * 4 + w.B * w.H * (2 * w.d_k + 2 * w.d_v) * 2


def backward_flops(w):
    """Three chunkwise evaluations per gradient pass: (chunk_out share, chunk_dS share)."""
    b, n = w.chunk, w.B * w.H * w.L
    return 3 * n * (2 * b * (w.d_k + w.d_v) + 2 * w.d_k * w.d_v), 3 * n * 2 * w.d_k * w.d_v


def backward_tc_bytes(w, grad_bytes=2):
    """Bytes the HBM-bound kernels of the tensor-core gradient pass move per
    step: the operand layouts (bwd_prep: q, k, v, dO read once; ω·dO, ζ·V,
    K̂′ and Q″ padded to whole chunks, K′ and Q′ unpadded) and the gradients
    dq, dk (bwd_grad_out: the piece outputs, in the gradients' type, in;
    gradients out; dv is written by the chunk kernel itself)."""
    n = w.B * w.H
    Lp = -(-w.L // 128) * 128
    P = -(-w.d_v // 256)
    rd = n * w.L * 2 * (2 * w.d_v + 2 * w.d_k)
    wr = n * 2 * (2 * Lp * w.d_v + 2 * w.L * w.d_k + 2 * Lp * w.d_k)
    go = n * w.L * 2 * (P * w.d_k * grad_bytes + w.d_k * grad_bytes)
    return {"bwd_prep": rd + wr, "bwd_grad_out": go}


def param_walk_bytes(w):
    """Bytes the two tensor-core state walks of ret_chunkwise_param_grads move
    per call (bf16 inputs): forward, v and kf (bf16 hi + lo, rows padded to
    whole chunks) in, S_in in, the per-chunk fp32 states out; backward, dO
    and qb in, the states, S_in and dS_out in."""
    n = w.B * w.H
    Lp = -(-w.L // 128) * 128
    C = Lp // 128
    rows = n * w.L * w.d_v * 2
    ops = n * Lp * w.d_k * 4
    state = n * w.d_k * w.d_v * 4
    return (rows + ops + state + C * state) + (rows + ops + C * state + 2 * state)


# fp32 FFMA peak: 148 SMs x 128 fp32 lanes x 2 flop per FFMA at the 2032 MHz maximum SM clock.
FFMA_TFLOPS = 148 * 128 * 2 * 2032e6 / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


CHUNK_KERNEL_FILES = ("kernel_tc_pair.cuh", "kernel_tc_chunk.cuh", "tc_primitives.cuh", "common.cuh")


def kernel_source_sha(files=CHUNK_KERNEL_FILES):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "linear_recurrent_sequence_prologue_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload="msr7b", files=CHUNK_KERNEL_FILES):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m1 = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    m2 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m1 or not m2 or m1.group(1) != kernel_source_sha(files):
        return None
    return float(m2.group(1))


# --------------------------------------------------------------------------
# Multi-rank timing: one independent replica per rank (the path has no
# exchange step); the job's time is the slowest rank's, its throughput the
# units of all ranks over that time.
# --------------------------------------------------------------------------
def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """Largest value of `value` over the ranks of the default process group."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job units per second when every rank processes units_per_rank."""
    return world * units_per_rank / seconds_max


def sustained_window(step, stream, dev_index, work, unit, peak, seconds=1.0):
    """The same step repeated for at least `seconds` right after the timed
    region, with its own device time and clock record: how the step runs once
    the GPU has settled under this load (the power cap of the part can lower
    the SM clock within a second).  Work per step in `unit` × 1e12 (TFLOP/s)
    or 1e9 (GB/s); compared with the sustained peak when one is given."""
    import torch
    sampler = ClockSampler(dev_index)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        sampler.mark()
        s.record(stream)
        n = soak(step, torch.cuda.synchronize, seconds)
        e.record(stream)
        torch.cuda.synchronize()
        sampler.mark()
    ms = s.elapsed_time(e) / n
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    ach = work / (ms / 1e3) / scale
    out = {"ms_per_step": ms, "steps": n, "achieved": ach, "unit": unit,
           "clocks": sampler.summary(),
           "note": "the step repeated for >= 1 s after the timed region (synchronised every 16 "
                   "steps), device time over all of them"}
    if peak:
        out["peak"] = peak
        out["frac"] = ach / peak
    return out


def soak(step, sync, seconds=1.0, batch=16):
    """Run `step` (untimed) for at least `seconds` of wall clock, synchronising
    every `batch` calls so that host time tracks device time; the clock
    sampler runs through it, so the record covers a second of this load."""
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds:
        for _ in range(batch):
            step()
        n += batch
        sync()
    return n


# --------------------------------------------------------------------------
# Clock sampling during the timed region (NVML reads only)
# --------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the timed region
    runs: through NVML when pynvml is importable, else by polling nvidia-smi
    (reads only; no GPU setting is touched)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, dev_index, period_s=0.002):
        self.samples, self.reasons, self.err, self.marks = [], set(), None, []
        self.nvml_error = None
        self.dev, self.period, self.max_mhz, self.source = dev_index, period_s, None, None
        self._stop = threading.Event()
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(dev_index)
            self._reasons_fn = (getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
                                or getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons"))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
        except Exception as e:  # noqa: BLE001
            self.nvml_error = f"{type(e).__name__}: {e}"
            import shutil
            if shutil.which("nvidia-smi"):
                self.source = "nvidia-smi"
            else:
                self.err = self.nvml_error

    def mark(self):
        """Record the current sample count (start / end of the timed region)."""
        self.marks.append(len(self.samples))

    def _sample_nvml(self):
        self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
        bits = int(self._reasons_fn(self.h))
        self.reasons |= {n for b, n in self.REASONS.items() if bits & b}

    def _sample_smi(self):
        import subprocess
        out = subprocess.run(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + ",".join(self.SMI_FIELDS),
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=5).stdout.strip().split(",")
        vals = [v.strip() for v in out]
        self.samples.append(float(vals[0]))
        self.max_mhz = float(vals[1])
        for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                            "sw_power_cap"), vals[2:]):
            if v.lower() == "active":
                self.reasons.add(name)

    def _sample(self):
        (self._sample_nvml if self.source == "nvml" else self._sample_smi)()

    def _run(self):
        while not self._stop.is_set():
            try:
                self._sample()
            except Exception as e:  # noqa: BLE001
                self.err = f"{type(e).__name__}: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.source:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.source:
            self._stop.set()
            self.t.join()

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples), "source": self.source}
        if len(self.marks) >= 2:
            inside = self.samples[self.marks[0]:self.marks[1] + 1]
            out["samples_in_timed_region"] = len(inside)
            if inside:
                out["sm_mhz_timed_region"] = statistics.median(inside)
            out["window"] = "samples from the sampler's start through the end of the timed region"
        if self.err:
            out["error"] = self.err
        if self.nvml_error and self.source != "nvml":
            out["nvml_unavailable"] = self.nvml_error
        return out


# --------------------------------------------------------------------------
# CPU baseline: the float64 oracle as it stands, on a bounded sample
# --------------------------------------------------------------------------
def cpu_baseline(w, inp, budget_s=12.0):
    import numpy as np
    from oracle import retention_ref as O
    from linear_recurrent_sequence_prologue_b300.inputs import to_f64
    try:
        from threadpoolctl import threadpool_info
        cores = max([d.get("num_threads", 1) for d in threadpool_info()] or [1])
    except Exception:
        cores = os.cpu_count()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done, t0 = 0, time.perf_counter()
    for b, h in heads:
        sl = lambda t: to_f64(t[b:b + 1, h:h + 1])
        O.retention(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                    np.asarray(inp["gamma"], np.float64)[h:h + 1],
                    np.asarray(inp["theta"], np.float64), 0,
                    None if inp["state_in"] is None else sl(inp["state_in"]), "chunkwise", w.chunk)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    per_head = dt / done
    value = (w.B * w.L) / (per_head * len(heads))
    out = {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{done} of {len(heads)} (b,h) heads of the {w.name} workload, float64 "
                     f"chunkwise oracle, {dt:.1f} s; tokens/s scaled to all heads"}
    # the same oracle on one thread, on at most two heads (a few seconds)
    try:
        from threadpoolctl import threadpool_limits
        with threadpool_limits(limits=1):
            done1, t1 = 0, time.perf_counter()
            for b, h in heads[:2]:
                sl = lambda t: to_f64(t[b:b + 1, h:h + 1])
                O.retention(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                            np.asarray(inp["gamma"], np.float64)[h:h + 1],
                            np.asarray(inp["theta"], np.float64), 0,
                            None if inp["state_in"] is None else sl(inp["state_in"]), "chunkwise",
                            w.chunk)
                done1 += 1
                if time.perf_counter() - t1 > budget_s / 3:
                    break
            dt1 = time.perf_counter() - t1
        out["value_1_thread"] = (w.B * w.L) / (dt1 / done1 * len(heads))
        out["sample_1_thread"] = f"{done1} head(s) on 1 thread, {dt1:.1f} s; scaled to all heads"
    except ImportError:
        pass
    return out


# --------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from linear_recurrent_sequence_prologue_b300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=0)
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, inp, budget_s=2.0)
        if i >= args.warmup:
            vals.append(r["value"])
    v = statistics.median(vals)
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "impl": "reference",
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d_k": w.d_k,
                       "d_v": w.d_v, "chunk": w.chunk},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"] + " (per step)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "vs_baseline": None}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.profile:
        return run_profile_case(args.profile)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from linear_recurrent_sequence_prologue_b300 import build
    build.build()
    import linear_recurrent_sequence_prologue_b300 as R
    from linear_recurrent_sequence_prologue_b300 import _lib
    from linear_recurrent_sequence_prologue_b300.inputs import (WORKLOADS, make_decode_inputs,
                                                                make_inputs)
    lib = R.load()
    peaks, peak_kind = measured_peaks()
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=0)
    q, k, v = inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev)
    s_in = inp["state_in"].to(dev) if inp["state_in"] is not None else None
    out = torch.empty((w.B, w.H, w.L, w.d_v), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty((w.B, w.H, w.d_k, w.d_v), dtype=torch.float32, device=dev)
    _, ws_bytes = R.plan("chunkwise", torch.bfloat16, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk,
                         gamma=inp["gamma"])
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    def time_launches(fn, n, warm=3):
        """Average device time of one fn() call (CUDA events on the launching
        stream, synchronised on both sides, after warm-up calls)."""
        for _ in range(warm):
            if fn() != _lib.RET_OK:
                raise RuntimeError("warm-up call failed")
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    # The timed loop calls the C ABI directly with arguments marshalled once,
    # so host-side Python work cannot leave gaps between launches.
    import ctypes as C
    garr = np.ascontiguousarray(inp["gamma"], np.float32)
    tarr = np.ascontiguousarray(inp["theta"], np.float32)
    fptr = lambda a: a.ctypes.data_as(C.POINTER(C.c_float))
    vp = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    cargs = (vp(q), vp(k), vp(v), _lib.RET_BF16, fptr(garr), fptr(tarr), w.B, w.H, w.L, w.d_k,
             w.d_v, 0, w.chunk, vp(s_in), None, vp(out), _lib.RET_BF16, None, vp(ws), ws_bytes,
             C.c_void_p(stream.cuda_stream))

    def cstep():
        st = lib.ret_chunkwise(*cargs)
        if st != _lib.RET_OK:
            raise RuntimeError(f"ret_chunkwise returned {st}")

    for _ in range(args.warmup):
        cstep()
    torch.cuda.synchronize()

    # Per-launch events through the library's profiling hook, armed for the
    # first steps of the timed region (it records at most 64 launches).
    hook_steps = min(args.steps, 16)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(128)]
    for e in evs:   # torch creates CUDA events lazily; record once to materialise
        e.record(stream)
    torch.cuda.synchronize()
    ev_handles = (C.c_void_p * len(evs))(*[C.c_void_p(e.cuda_event) for e in evs])

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    with sampler:
        sampler.mark()
        start.record(stream)
        lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
        for it in range(args.steps):
            cstep()
            if it + 1 == hook_steps:
                n_k = lib.ret_profile_end()
        end.record(stream)
        torch.cuda.synchronize()
        sampler.mark()
    names = [lib.ret_profile_kernel(i).decode() for i in range(n_k)]
    barrier()
    ms = start.elapsed_time(end)
    sustained = sustained_window(cstep, stream, local, chunk_flops(w), "TFLOP/s",
                                 peaks.get("bf16_tflops_sustained"))
    per_kernel = {}
    for i, nm in enumerate(names):
        per_kernel.setdefault(nm, []).append(evs[2 * i].elapsed_time(evs[2 * i + 1]))
    launches_per_step = n_k / hook_steps
    ms = max_over_ranks(ms, world, dev)
    tok_per_step = w.B * w.L
    value = replica_throughput(tok_per_step * args.steps, ms / 1e3, world)
    flops = chunk_flops(w)
    top = max(per_kernel, key=lambda n: sum(per_kernel[n]))
    top_ms = statistics.mean(per_kernel[top])
    achieved = flops / (top_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = profiled_traffic(top)

    # ---------------- the same call in the compact-workspace mode ----------------
    # For comparison: ret_chunkwise given only ret_chunkwise_plan_compact's
    # workspace runs the Θ prologue inside the chunk launch (producer CTAs
    # and an L2-resident ring) instead of the front pass.
    def compact_line(steps=20):
        _, cb = R.plan("chunkwise_compact", torch.bfloat16, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk,
                       gamma=inp["gamma"])
        if cb >= ws_bytes:
            return None
        cws_ = torch.empty(max(cb, 1), dtype=torch.uint8, device=dev)
        fargs = list(cargs)
        fargs[18], fargs[19] = vp(cws_), cb

        def fstep():
            st_ = lib.ret_chunkwise(*fargs)
            if st_ != _lib.RET_OK:
                raise RuntimeError(f"ret_chunkwise (compact workspace) returned {st_}")

        for _ in range(3):
            fstep()
        torch.cuda.synchronize()
        fs_, fe_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fs_.record(stream)
        lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
        for i_ in range(steps):
            fstep()
            if i_ + 1 == 8:
                nf = lib.ret_profile_end()
        fe_.record(stream)
        torch.cuda.synchronize()
        fper = {}
        for i_ in range(nf):
            fper.setdefault(lib.ret_profile_kernel(i_).decode(), []).append(
                evs[2 * i_].elapsed_time(evs[2 * i_ + 1]))
        del cws_
        return {"ms_per_step": fs_.elapsed_time(fe_) / steps, "steps": steps, "workspace_bytes": cb,
                "kernels_ms": {n: statistics.mean(t) for n, t in fper.items()},
                "note": "ret_chunkwise with ret_chunkwise_plan_compact's workspace: the rotation "
                        "inside the chunk launch (producer CTAs, L2 ring), for comparison"}

    compact = compact_line()

    # ---------------- the Small and 1.3B-shape workloads ----------------
    def bench_config(name, steps):
        """Time ret_chunkwise on one more workload: tokens/s, per-kernel times and
        a roofline (the HBM bound for Small, whose arithmetic intensity is below
        the ridge; the bf16 peak for the 1.3B shape).  Inputs smaller than L2 are
        replicated into enough copies that consecutive steps read different
        ones and the copies together exceed twice the 126 MB L2."""
        cw = WORKLOADS[name]
        cin = make_inputs(cw, seed=0)
        in_bytes = sum(cin[n].numel() * cin[n].element_size() for n in ("q", "k", "v"))
        copies = max(1, -(-2 * 126 * 2 ** 20 // in_bytes))
        sets = [tuple(cin[n].to(dev) for n in ("q", "k", "v")) for _ in range(copies)]
        cs_in = cin["state_in"].to(dev) if cin["state_in"] is not None else None
        couts = [torch.empty((cw.B, cw.H, cw.L, cw.d_v), dtype=torch.bfloat16, device=dev)
                 for _ in range(copies)]
        cs_out = torch.empty((cw.B, cw.H, cw.d_k, cw.d_v), dtype=torch.float32, device=dev)
        cpath, cws_bytes = R.plan("chunkwise", torch.bfloat16, cw.B, cw.H, cw.L, cw.d_k, cw.d_v,
                                  cw.chunk, gn=cw.groupnorm, gamma=cin["gamma"])
        cws = torch.empty(max(cws_bytes, 1), dtype=torch.uint8, device=dev)
        cg = np.ascontiguousarray(cin["gamma"], np.float32)
        ct = np.ascontiguousarray(cin["theta"], np.float32)
        gns = _lib.RetGN(1, cw.gn_eps, None, None) if cw.groupnorm else None
        gnp = C.byref(gns) if gns is not None else None
        cargs_ = [(vp(a), vp(b), vp(c_), _lib.RET_BF16, fptr(cg), fptr(ct), cw.B, cw.H, cw.L,
                   cw.d_k, cw.d_v, 0, cw.chunk, vp(cs_in), vp(cs_out), vp(o_), _lib.RET_BF16, gnp,
                   vp(cws), cws_bytes, C.c_void_p(stream.cuda_stream))
                  for (a, b, c_), o_ in zip(sets, couts)]
        it_ = [0]

        def one():
            st_ = lib.ret_chunkwise(*cargs_[it_[0] % copies])
            it_[0] += 1
            if st_ != _lib.RET_OK:
                raise RuntimeError(f"ret_chunkwise ({name}) returned {st_}")

        for _ in range(max(3, args.warmup)):
            one()
        torch.cuda.synchronize()
        hook = min(steps, 8)
        csampler = ClockSampler(local)
        cs_, ce_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        with csampler:
            csampler.mark()
            cs_.record(stream)
            lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
            for i_ in range(steps):
                one()
                if i_ + 1 == hook:
                    nk_ = lib.ret_profile_end()
            ce_.record(stream)
            torch.cuda.synchronize()
            csampler.mark()
        cnames = [lib.ret_profile_kernel(i).decode() for i in range(nk_)]
        cper = {}
        for i_, nm in enumerate(cnames):
            cper.setdefault(nm, []).append(evs[2 * i_].elapsed_time(evs[2 * i_ + 1]))
        cms = max_over_ranks(cs_.elapsed_time(ce_) / steps, world, dev)
        cstep_ms = {nm: sum(t) / hook for nm, t in cper.items()}
        ctop = max(cstep_ms, key=cstep_ms.get)
        cfl, cby = chunk_flops(cw), chunk_bytes(cw)
        if name == "small":
            bound, pk, unit_ = "hbm", peaks["hbm_gbs"], "GB/s"
            ach = cby / (cms / 1e3) / 1e9
            knote = "whole call: algorithmic bytes / call time"
        else:
            bound, pk, unit_ = "tensor", peak, "TFLOP/s"
            ach = cfl / (cstep_ms[ctop] / 1e3) / 1e12
            knote = f"kernel {ctop}: algorithmic flop / its launch time"
        res = {"metric": "chunkwise retention tokens/s", "unit": "tokens/s",
               "value": replica_throughput(cw.B * cw.L, cms / 1e3, world), "ms_per_step": cms,
               "steps": steps, "path": "tensor cores" if cpath == _lib.RET_PATH_TC else "fp32 kernels",
               "config": {"workload": cw.name, "B": cw.B, "H": cw.H, "L": cw.L, "d_k": cw.d_k,
                          "d_v": cw.d_v, "chunk": cw.chunk, "groupnorm": cw.groupnorm,
                          "state_in": cs_in is not None, "input_copies": copies},
               "roofline": {"bound": bound, "achieved": ach, "peak": pk, "unit": unit_,
                            "frac": ach / pk, "note": knote, "traffic": None,
                            "peak_kind": peak_kind,
                            "algorithmic_flop_per_call": cfl, "algorithmic_bytes_per_call": cby,
                            "call_tflops": cfl / (cms / 1e3) / 1e12,
                            "call_frac_of_bf16_peak": cfl / (cms / 1e3) / 1e12 / peak},
               "kernels_ms_per_step": cstep_ms,
               "gpu_launches": int(round(nk_ / hook * steps)), "clocks": csampler.summary()}
        del sets, couts, cws
        return res

    extra = {}
    for name, steps_ in (("small", 200), ("msr1p3b", 50)):
        if name != w.name:
            extra[name] = bench_config(name, steps_)

    # ---------------- the MSR block around the core (projections, gate) ----------------
    def block_line(steps=10):
        """ret_msr_block at the 7B shape (hidden 4096, H16, d_k 256, d_v 512) with
        seeded random bf16 weights: tokens/s, TFLOP/s of the whole block and the
        roofline of its dominant kernel."""
        D, Dout = w.H * w.d_k, w.H * w.d_k
        HK, HV = w.H * w.d_k, w.H * w.d_v
        gen = torch.Generator(device=dev).manual_seed(11)
        rn = lambda shape, std: (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)
        xb = rn((w.B, w.L, D), 1.0)
        wq, wk = rn((D, w.H, w.d_k), D ** -0.5), rn((D, w.H, w.d_k), D ** -0.5)
        wv, wg = rn((D, w.H, w.d_v), D ** -0.5), rn((D, w.H, w.d_v), D ** -0.5)
        wo = rn((w.H, w.d_v, Dout), HV ** -0.5)
        zb = torch.empty((w.B, w.L, Dout), dtype=torch.bfloat16, device=dev)
        sb_ = torch.empty((w.B, w.H, w.d_k, w.d_v), dtype=torch.float32, device=dev)
        nbytes = R.msr_block_plan(w.B, w.L, D, w.H, w.d_k, w.d_v, Dout, gamma=inp["gamma"])
        bws_ = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        bargs_ = (vp(xb), vp(wq), vp(wk), vp(wv), vp(wg), vp(wo), fptr(garr), fptr(tarr), w.B, w.L, D, w.H,
                  w.d_k, w.d_v, Dout, 0, vp(s_in), vp(sb_), vp(zb), _lib.RET_BF16, 1e-5, vp(bws_), nbytes,
                  C.c_void_p(stream.cuda_stream))

        def one():
            st_ = lib.ret_msr_block(*bargs_)
            if st_ != _lib.RET_OK:
                raise RuntimeError(f"ret_msr_block returned {st_}")

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        bsamp = ClockSampler(local)
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with bsamp:
            bsamp.mark()
            s0.record(stream)
            lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
            for i_ in range(steps):
                one()
                if i_ == 1:
                    nk_ = lib.ret_profile_end()
            e0.record(stream)
            torch.cuda.synchronize()
            bsamp.mark()
        bper = {}
        for i_ in range(nk_):
            bper.setdefault(lib.ret_profile_kernel(i_).decode(), []).append(evs[2 * i_].elapsed_time(evs[2 * i_ + 1]))
        step_ms = {nm: sum(t) / 2 for nm, t in bper.items()}
        bms_ = max_over_ranks(s0.elapsed_time(e0) / steps, world, dev)
        M = w.B * w.L
        gemm_fl = {"proj_q_rot": 2 * M * D * HK, "proj_k_rot": 2 * M * D * HK, "proj_v": 2 * M * D * HV,
                   "proj_gate": 2 * M * D * HV, "proj_out": 2 * M * HV * Dout}
        total = sum(gemm_fl.values()) + chunk_flops(w)
        gtop = max(gemm_fl, key=lambda n: step_ms.get(n, 0.0))
        gach = gemm_fl[gtop] / (step_ms[gtop] / 1e3) / 1e12
        del bws_, xb, wq, wk, wv, wg, wo, zb
        return {"metric": "MSR block tokens/s", "value": replica_throughput(M, bms_ / 1e3, world),
                "unit": "tokens/s", "ms_per_step": bms_, "steps": steps,
                "config": {"workload": "msr7b block", "B": w.B, "L": w.L, "hidden": D, "H": w.H, "d_k": w.d_k,
                           "d_v": w.d_v, "D_out": Dout, "weights": "seeded random bf16, N(0, 1/fan_in)"},
                "tflops": total / (bms_ / 1e3) / 1e12, "frac_of_bf16_peak": total / (bms_ / 1e3) / 1e12 / peak,
                "algorithmic_flop_per_step": total,
                "roofline": {"bound": "tensor", "kernel": gtop, "achieved": gach, "peak": peak,
                             "unit": "TFLOP/s", "frac": gach / peak, "traffic": None,
                             "algorithmic_flop_per_launch": gemm_fl[gtop]},
                "kernels_ms_per_step": step_ms,
                "gpu_launches": int(round(nk_ / 2 * steps)), "clocks": bsamp.summary()}

    block = block_line()

    # ---------------- decode workload ----------------
    dw = WORKLOADS["decode"]
    dsteps = max(args.decode_steps, 1)
    pool = 16
    dinp = make_decode_inputs(dw, seed=0, steps=pool, device=f"cuda:{local}")
    dstate = dinp["state"]
    dout = torch.empty((dw.B, dw.H, dw.d_v), dtype=torch.bfloat16, device=dev)

    dg = np.ascontiguousarray(dinp["gamma"], np.float32)
    dth = np.ascontiguousarray(dinp["theta"], np.float32)
    dptrs = [(vp(dinp["q"][i]), vp(dinp["k"][i]), vp(dinp["v"][i])) for i in range(pool)]
    dstream = C.c_void_p(stream.cuda_stream)

    def dstep(t):
        qp_, kp_, vp_ = dptrs[t % pool]
        st = lib.ret_step(qp_, kp_, vp_, _lib.RET_BF16, fptr(dg), fptr(dth), dw.B, dw.H, dw.d_k,
                          dw.d_v, t, vp(dstate), vp(dout), _lib.RET_BF16, None, dstream)
        if st != _lib.RET_OK:
            raise RuntimeError(f"ret_step returned {st}")

    for t in range(max(3, args.warmup)):
        dstep(t)
    torch.cuda.synchronize()
    ds, de = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dsampler = ClockSampler(local)
    barrier()
    with dsampler:
        dsampler.mark()
        ds.record(stream)
        for t in range(dsteps):
            dstep(t)
        de.record(stream)
        torch.cuda.synchronize()
        dsampler.mark()
    dms = max_over_ranks(ds.elapsed_time(de) / dsteps, world, dev)
    dsus = sustained_window(lambda: dstep(0), stream, local, decode_bytes(dw), "GB/s",
                            peaks["hbm_gbs"])
    dgbs = decode_bytes(dw) / (dms / 1e3) / 1e9
    decode = {"metric": "decode state GB/s", "value": replica_throughput(dgbs, 1.0, world), "unit": "GB/s",
              "ms_per_step": dms, "steps": dsteps,
              "config": {"workload": "decode", "B": dw.B, "H": dw.H, "d_k": dw.d_k, "d_v": dw.d_v,
                         "state_bytes": 4 * dw.B * dw.H * dw.d_k * dw.d_v,
                         "l2": "state 1.07 GB > 126 MB L2 (no flush needed)"},
              "roofline": {"bound": "hbm", "achieved": dgbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": dgbs / peaks["hbm_gbs"],
                           "traffic": profiled_traffic("decode_step", "decode",
                                                       ("kernels_simt.cuh", "common.cuh")),
                           "peak_kind": peak_kind},
              "gpu_launches": dsteps, "clocks": dsampler.summary(), "sustained": dsus}
    del dinp, dstate

    # ---------------- row-normalised decay variant on the chunkwise output ----------------
    nsteps = 20
    garr_c = fptr(garr)
    for _ in range(3):
        lib.ret_decay_row_norm(vp(out), _lib.RET_BF16, garr_c, w.B, w.H, w.L, w.d_v, 0,
                               C.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    ns_, ne_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ns_.record(stream)
    for _ in range(nsteps):
        st_ = lib.ret_decay_row_norm(vp(out), _lib.RET_BF16, garr_c, w.B, w.H, w.L, w.d_v, 0,
                                     C.c_void_p(stream.cuda_stream))
        if st_ != _lib.RET_OK:
            raise RuntimeError(f"ret_decay_row_norm returned {st_}")
    ne_.record(stream)
    torch.cuda.synchronize()
    nms = ns_.elapsed_time(ne_) / nsteps
    nbytes = 2 * w.B * w.H * w.L * w.d_v * 2   # read and write the bf16 output
    ngbs = nbytes / (nms / 1e3) / 1e9
    row_norm = {"metric": "row-normalised decay pass GB/s", "value": ngbs, "unit": "GB/s",
                "ms_per_launch": nms, "launches": nsteps,
                "roofline": {"bound": "hbm", "achieved": ngbs, "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": ngbs / peaks["hbm_gbs"], "traffic": None,
                             "algorithmic_bytes_per_launch": nbytes}}

    # ---------------- gradient pass (fp32 kernels) on the same workload ----------------
    backward = None
    if args.backward_steps > 0:
        from linear_recurrent_sequence_prologue_b300.inputs import make_grad_inputs
        gi = make_grad_inputs(w, seed=5, d_state_std=1.0)
        d_o, dso = gi["d_out"].to(dev), gi["d_state_out"].to(dev)
        grads = tuple(torch.empty_like(t) for t in (q, k, v))
        dsi = torch.empty_like(dso)
        bpath, bws_bytes = R.backward_plan(torch.bfloat16, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk,
                                           gamma=inp["gamma"])
        bws = torch.empty(bws_bytes, dtype=torch.uint8, device=dev)
        bargs = (vp(q), vp(k), vp(v), vp(d_o), _lib.RET_BF16, fptr(garr), fptr(tarr), w.B, w.H, w.L,
                 w.d_k, w.d_v, 0, w.chunk, vp(s_in), vp(dso), vp(grads[0]), vp(grads[1]),
                 vp(grads[2]), _lib.RET_BF16, vp(dsi), vp(bws), bws_bytes, C.c_void_p(stream.cuda_stream))

        def bstep():
            st = lib.ret_chunkwise_backward(*bargs)
            if st != _lib.RET_OK:
                raise RuntimeError(f"ret_chunkwise_backward returned {st}")

        for _ in range(max(3, args.warmup)):
            bstep()
        torch.cuda.synchronize()
        bs, be = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        bsampler = ClockSampler(local)
        bhook = min(args.backward_steps, 2)
        barrier()
        with bsampler:
            bs.record(stream)
            lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
            for it in range(args.backward_steps):
                bstep()
                if it + 1 == bhook:
                    nb_k = lib.ret_profile_end()
            be.record(stream)
            torch.cuda.synchronize()
        bnames = [lib.ret_profile_kernel(i).decode() for i in range(nb_k)]
        bper = {}
        for i, nm in enumerate(bnames):
            bper.setdefault(nm, []).append(evs[2 * i].elapsed_time(evs[2 * i + 1]))
        bms = max_over_ranks(bs.elapsed_time(be) / args.backward_steps, world, dev)
        f_out, f_ds = backward_flops(w)
        step_ms = {nm: sum(t) / bhook for nm, t in bper.items()}   # all launches of a name, per step
        btop = max(step_ms, key=step_ms.get)
        bbytes = None
        if bpath == _lib.RET_PATH_TC:
            # the chunk kernels run all four products of the three evaluations;
            # the operand and gradient passes are HBM-bound
            bflops = {"bwd_chunk_tc": f_out + f_ds}.get(btop)
            bbytes = backward_tc_bytes(w).get(btop)
            if bflops:
                bpeak, bbound, bkind = peak, "tensor", f"bf16_tflops burst ({peak_kind})"
            else:
                bpeak, bbound, bkind = peaks["hbm_gbs"], "hbm", f"hbm_gbs ({peak_kind})"
            bdt = "bf16 (bf16 operands, fp32 accumulation; bf16 gradients)"
        else:
            bflops = {"bwd_chunk_out": f_out, "bwd_chunk_dS": f_ds}.get(btop)
            bpeak, bbound = FFMA_TFLOPS, "alu"
            bkind = "derived: 148 SMs x 128 fp32 lanes x 2 flop x 2032 MHz"
            bdt = "f32 (bf16 inputs and gradients)"
        if bflops:
            bach = bflops / (step_ms[btop] / 1e3) / 1e12
        elif bbytes:
            bach = bbytes / (step_ms[btop] / 1e3) / 1e9
        else:
            bach = None
        backward = {
            "metric": "gradient pass tokens/s", "value": replica_throughput(w.B * w.L, bms / 1e3, world),
            "unit": "tokens/s", "ms_per_step": bms, "steps": args.backward_steps,
            "dtype": bdt, "path": "tensor cores" if bpath == _lib.RET_PATH_TC else "fp32 kernels",
            "config": {"workload": w.name, "chunk": w.chunk, "state_in": True, "d_state_out": True},
            "roofline": {"bound": bbound, "kernel": btop, "achieved": bach, "peak": bpeak,
                         "unit": "GB/s" if bbound == "hbm" else "TFLOP/s",
                         "frac": bach / bpeak if bach else None,
                         "traffic": None, "peak_kind": bkind,
                         "algorithmic_flop_per_step": f_out + f_ds,
                         "algorithmic_bytes_of_kernel_per_step": bbytes},
            "kernels_ms_per_step": step_ms,
            "gpu_launches": int(round(nb_k / bhook * args.backward_steps)),
            "clocks": bsampler.summary()}

        # γ and θ gradients from this forward (out, s_out) and backward (grads, dsi):
        # two HBM-bound row passes over 8 token-major tensors plus the states
        pws_n = C.c_size_t(0)
        lib.ret_chunkwise_param_grads_plan(w.B, w.H, w.L, w.d_k, w.d_v, C.byref(pws_n))
        pws = torch.empty(max(pws_n.value, 1), dtype=torch.uint8, device=dev)
        dgam = torch.empty(w.H, dtype=torch.float32, device=dev)
        dthe = torch.empty(w.d_k // 2, dtype=torch.float32, device=dev)
        pargs = (vp(q), vp(k), vp(v), vp(d_o), _lib.RET_BF16, vp(out), _lib.RET_BF16, vp(grads[0]),
                 vp(grads[1]), vp(grads[2]), _lib.RET_BF16, fptr(garr), fptr(tarr), w.B, w.H, w.L, w.d_k,
                 w.d_v, 0, vp(s_in), vp(dso), vp(dgam), vp(dthe), vp(pws), pws_n.value,
                 C.c_void_p(stream.cuda_stream))
        lib.ret_profile_begin(C.cast(ev_handles, C.c_void_p), len(evs))
        if lib.ret_chunkwise_param_grads(*pargs) != _lib.RET_OK:
            raise RuntimeError("ret_chunkwise_param_grads failed")
        np_k = lib.ret_profile_end()
        torch.cuda.synchronize()
        pker = {}
        for i in range(np_k):
            nm = lib.ret_profile_kernel(i).decode()
            pker[nm] = pker.get(nm, 0.0) + evs[2 * i].elapsed_time(evs[2 * i + 1])
        pms = time_launches(lambda: lib.ret_chunkwise_param_grads(*pargs), 10)
        tok = w.B * w.H * w.L
        walk_ms = pker.get("param_walk_fwd", 0.0) + pker.get("param_walk_bwd", 0.0)
        wbytes = param_walk_bytes(w)
        wgbs = wbytes / (walk_ms / 1e3) / 1e9 if walk_ms else None
        rbytes = tok * (4 * w.d_v + 4 * w.d_k) * 2
        rgbs = rbytes / (pker["param_rows"] / 1e3) / 1e9 if pker.get("param_rows") else None
        backward["param_grads"] = {
            "metric": "gamma/theta gradient call ms", "value": pms, "unit": "ms", "ms_per_call": pms,
            "launches_per_call": np_k, "kernels_ms": pker,
            # the tensor-core walks stream their operands and the per-chunk states
            "roofline": {"bound": "hbm", "kernel": "param_walk_fwd + param_walk_bwd",
                         "achieved": wgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": wgbs / peaks["hbm_gbs"] if wgbs else None, "traffic": None,
                         "peak_kind": f"hbm_gbs ({peak_kind})",
                         "algorithmic_bytes_per_call": wbytes,
                         "walk_flop_per_call": 2 * 2 * 2 * tok * w.d_k * w.d_v},
            "row_pass": {"algorithmic_bytes": rbytes, "achieved_gbs": rgbs,
                         "frac_of_hbm": rgbs / peaks["hbm_gbs"] if rgbs else None}}
        del pws, dgam, dthe
        del bws, grads, dsi, d_o, dso, gi

        # GroupNorm backward at the 1.3B shape (bf16 rows of 512 channels, with weight)
        gw_ = WORKLOADS["msr1p3b"]
        gg = torch.Generator(device=dev).manual_seed(12)
        gx = torch.randn((gw_.B, gw_.H, gw_.L, gw_.d_v), generator=gg, device=dev).to(torch.bfloat16)
        gdy = torch.randn((gw_.B, gw_.H, gw_.L, gw_.d_v), generator=gg, device=dev).to(torch.bfloat16)
        gwt = torch.randn((gw_.H, gw_.d_v), generator=gg, device=dev)
        gdx = torch.empty_like(gx)
        gdw, gdb = torch.empty_like(gwt), torch.empty_like(gwt)
        gws_n = C.c_size_t(0)
        lib.ret_groupnorm_backward_plan(gw_.B, gw_.H, gw_.L, gw_.d_v, C.byref(gws_n))
        gws = torch.empty(gws_n.value, dtype=torch.uint8, device=dev)
        gargs = (vp(gx), vp(gdy), _lib.RET_BF16, vp(gwt), C.c_float(1e-5), gw_.B, gw_.H, gw_.L, gw_.d_v,
                 vp(gdx), _lib.RET_BF16, vp(gdw), vp(gdb), vp(gws), gws_n.value, C.c_void_p(stream.cuda_stream))
        gms = time_launches(lambda: lib.ret_groupnorm_backward(*gargs), 20)
        gbytes = 3 * gx.numel() * 2 + gws_n.value
        ggbs = gbytes / (gms / 1e3) / 1e9
        backward["groupnorm_backward"] = {
            "metric": "GroupNorm backward GB/s", "value": ggbs, "unit": "GB/s", "ms_per_call": gms,
            "config": {"workload": gw_.name, "B": gw_.B, "H": gw_.H, "L": gw_.L, "d_v": gw_.d_v,
                       "dtype": "bf16 x, dy, dx; fp32 weight and parameter gradients"},
            "launches_per_call": 2, "algorithmic_bytes_per_call": gbytes,
            "roofline": {"bound": "hbm", "achieved": ggbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ggbs / peaks["hbm_gbs"], "traffic": None}}
        del gx, gdy, gwt, gdx, gdw, gdb, gws

    # ---------------- end to end through the API with host buffers ----------------
    # Every step copies its inputs host → device from pinned memory, runs
    # ret_chunkwise through the Python API and copies out and state_out back.
    # Steps are pipelined over two device buffer sets: the copy-in of step
    # k+1 and the copy-out of step k run on their own streams (separate copy
    # engines) while step k+1 computes; events order each buffer's reuse.
    hq, hk, hv = inp["q"].pin_memory(), inp["k"].pin_memory(), inp["v"].pin_memory()
    hs = inp["state_in"].pin_memory() if inp["state_in"] is not None else None
    hout = torch.empty((w.B, w.H, w.L, w.d_v), dtype=torch.bfloat16).pin_memory()
    hsout = torch.empty((w.B, w.H, w.d_k, w.d_v), dtype=torch.float32).pin_memory()
    s_in_ = torch.cuda.Stream(device=dev)
    s_out_ = torch.cuda.Stream(device=dev)
    bufs = []
    for _ in range(2):
        bufs.append({
            "q": torch.empty_like(hq, device=dev), "k": torch.empty_like(hk, device=dev),
            "v": torch.empty_like(hv, device=dev),
            "s": torch.empty_like(hs, device=dev) if hs is not None else None,
            "o": torch.empty((w.B, w.H, w.L, w.d_v), dtype=torch.bfloat16, device=dev),
            "so": torch.empty((w.B, w.H, w.d_k, w.d_v), dtype=torch.float32, device=dev),
            "loaded": torch.cuda.Event(), "computed": torch.cuda.Event(), "stored": torch.cuda.Event(),
            "used": False})

    def e2e_step(kstep):
        bb = bufs[kstep % 2]
        with torch.cuda.stream(s_in_):
            if bb["used"]:
                s_in_.wait_event(bb["computed"])      # step k−2 has read these inputs
            for name, host in (("q", hq), ("k", hk), ("v", hv), ("s", hs)):
                if host is not None:
                    bb[name].copy_(host, non_blocking=True)
            bb["loaded"].record(s_in_)
        stream.wait_event(bb["loaded"])
        if bb["used"]:
            stream.wait_event(bb["stored"])           # step k−2's outputs have been copied out
        R.chunkwise(bb["q"], bb["k"], bb["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                    state_in=bb["s"], out=bb["o"], state_out=bb["so"], workspace=ws, stream=stream)
        bb["computed"].record(stream)
        with torch.cuda.stream(s_out_):
            s_out_.wait_event(bb["computed"])
            hout.copy_(bb["o"], non_blocking=True)
            hsout.copy_(bb["so"], non_blocking=True)
            bb["stored"].record(s_out_)
        bb["used"] = True

    for kstep in range(2):
        e2e_step(kstep)
    torch.cuda.synchronize()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    es.record(s_in_)
    for kstep in range(args.e2e_steps):
        e2e_step(kstep)
    ee.record(s_out_)
    torch.cuda.synchronize()
    ems = max_over_ranks(es.elapsed_time(ee) / args.e2e_steps, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hs,) if hs is not None else ()))
    d2h = hout.numel() * hout.element_size() + hsout.numel() * hsout.element_size()
    # The host link alone: the same bytes as plain pinned copies, each direction
    # timed by itself on its copy stream (4 repetitions after one warm-up).
    def link_ms(fn, st):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(4):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 4

    def copy_in():
        with torch.cuda.stream(s_in_):
            for name, host in (("q", hq), ("k", hk), ("v", hv), ("s", hs)):
                if host is not None:
                    bufs[0][name].copy_(host, non_blocking=True)

    def copy_out():
        with torch.cuda.stream(s_out_):
            hout.copy_(bufs[0]["o"], non_blocking=True)
            hsout.copy_(bufs[0]["so"], non_blocking=True)

    def both():   # the two directions at once, as the pipelined steps run them
        copy_in()
        copy_out()

    def link_both_ms():
        both()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b_in, b_out = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in_)
        s_out_.wait_event(a)
        for _ in range(4):
            both()
        b_in.record(s_in_)
        b_out.record(s_out_)
        torch.cuda.synchronize()
        return max(a.elapsed_time(b_in), a.elapsed_time(b_out)) / 4

    h2d_ms, d2h_ms = link_ms(copy_in, s_in_), link_ms(copy_out, s_out_)
    both_ms = link_both_ms()
    e2e = {"value": replica_throughput(tok_per_step, ems / 1e3, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": ems, "steps": args.e2e_steps,
           "pipelined": "copy-in, compute and copy-out of consecutive steps overlap (two buffer sets)",
           "link": {"h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "h2d_gbs": h2d / (h2d_ms / 1e3) / 1e9,
                    "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9,
                    "both_directions_ms": both_ms,
                    "bound_ms": max(h2d_ms, d2h_ms, both_ms),
                    "frac": max(h2d_ms, d2h_ms, both_ms) / ems,
                    "note": "plain pinned copies of the same bytes: each direction alone, and both at "
                            "once on their two copy streams; with the steps pipelined the copies of "
                            "consecutive steps overlap, so the slowest of these bounds a step"}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0, 1.28^2) q,k,v; state_in N(0, 1e-2))",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d_k": w.d_k,
                       "d_v": w.d_v, "chunk": w.chunk, "state_in": True,
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs 537 MB > 126 MB L2 (no flush needed)"},
            "roofline": {"bound": "tensor", "kernel": top, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": f"bf16_tflops burst ({peak_kind})",
                         "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peak),
                         "algorithmic_flop_per_launch": flops,
                         "algorithmic_bytes_per_launch": chunk_bytes(w),
                         "launch_ms": top_ms,
                         "call_achieved": flops / (ms / args.steps / 1e3) / 1e12,
                         "call_frac": flops / (ms / args.steps / 1e3) / 1e12 / peak,
                         "call_note": "the whole ret_chunkwise call (every kernel it launches) "
                                      "against the same peak"},
            "kernels_ms": {n: statistics.mean(t) for n, t in per_kernel.items()},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": sampler.summary(),
            "sustained": sustained,
            "compact_workspace_mode": compact,
            "workspace_bytes": ws_bytes,
            "decode": decode,
            "msr_block": block,
            "small": extra.get("small"),
            "msr1p3b": extra.get("msr1p3b"),
            "backward": backward,
            "decay_row_norm": row_norm,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
