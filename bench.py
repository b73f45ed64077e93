#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

One call = one attn_fwd over the whole workload (every query row of every
head).  Default workload C4: causal GQA, bf16, Q [4,32,4096,128], K/V
[4,8,4096,128] -- the configuration the throughput target is quoted on.  A
timed step is a block of calls (enough for about 120 ms of device time, so
the clock sampler sees the GPU under load), each call bracketed by its own
CUDA events with L2 flushed before it; the step's time is the sum.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C1..C5]
    python bench.py --impl reference ...   # the float64 CPU oracle, bounded samples

Prints ONE JSON line (rank 0): the headline workload, and under "workloads"
every one of C1-C5 (timing, roofline fractions, and the whole output compared
with the float64 oracle, whose run over that workload is also the CPU
baseline).  Multi-GPU (torchrun): every rank runs an independent replica of
the workload (the forward has no exchange step); value = all ranks' FLOPs /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_forward_attn_gb300 import workloads as wl  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of GB300 dense fp16/bf16 tensor peak; ms/call"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20          # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attn_fwd_tc_dram_traffic.txt")
# --backward's default shapes; a trailing M: that workload's causal mask given as an
# explicit tril mask (attn_bwd_masked)
BWD_WORKLOADS = "C4,C4M,C2,C5"
KERNEL_SOURCES = [os.path.join(ROOT, "attention_forward_attn_gb300", "csrc", f)
                  for f in ("attn_tc.cu", "attn_vconv.cu", "ptx.cuh")]


# ------------------------------------------------------------------ work accounting

def nominal_flops(w) -> float:
    """The metric's formula: 4*B*Hq*L^2*D, halved for causal."""
    f = 4.0 * w.B * w.Hq * w.L * w.L * w.D
    return f / 2 if w.causal else f


def visible_keys_per_row(w, valid_len):
    """|J_i| for every row i of one (b, h) head, per batch: array [B, L]."""
    i = np.arange(w.L, dtype=np.int64)
    out = np.empty((w.B, w.L), dtype=np.int64)
    for b in range(w.B):
        kv = w.L if valid_len is None else int(min(max(int(valid_len[b]), 0), w.L))
        out[b] = np.minimum(kv, i + 1) if w.causal else kv
    return out


def algorithmic_flops(w, valid_len) -> float:
    """Only unmasked work: 4*D per visible (query, key) pair (QK^T and PV)."""
    return 4.0 * w.D * w.Hq * float(visible_keys_per_row(w, valid_len).sum())


def io_bytes(w) -> dict:
    e = 2
    q = w.B * w.Hq * w.L * w.D * e
    kv = 2 * w.B * w.Hkv * w.L * w.D * e
    o = q
    lse = w.B * w.Hq * w.L * 4
    vl = w.B * 4 if w.padded else 0
    return {"q": q, "kv": kv, "o": o, "lse": lse, "valid_len": vl}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source for this workload; else None."""
    try:
        text = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_sha256_16") != kernel_source_hash():
        return None
    key = "dram_bytes_per_launch_%s" % workload
    try:
        return float(fields[key])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            # raw samples (the JSON line carries their summary): ATTN_BENCH_OUT or bench_out/
            out = os.environ.get("ATTN_BENCH_OUT", os.path.join(ROOT, "bench_out"))
            os.makedirs(out, exist_ok=True)
            self.path = os.path.join(out, "clocks_bench_%d.csv" % os.getpid())
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (identity for one process)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_flops: float, max_seconds: float, world: int) -> float:
    """Whole-job TFLOP/s: the work of every replica over the slowest rank's time."""
    return per_rank_flops * world / max_seconds / 1e12


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_sample(w, q, k, v, vl, budget_s: float, rng, threads: int = 0):
    """Time the float64 oracle on a bounded random sample of query rows of the
    workload.  Returns (TFLOP/s in the metric's convention, details)."""
    import oracle
    code = wl.dtype_code(w.dtype)
    qd = oracle.decode(wl.bits(q), code)
    kd = oracle.decode(wl.bits(k), code)
    vd = oracle.decode(wl.bits(v), code)
    vln = None if vl is None else vl.numpy()
    keys = visible_keys_per_row(w, vln)                      # [B, L]
    total_rows = w.B * w.Hq * w.L
    ratio = nominal_flops(w) / max(algorithmic_flops(w, vln), 1.0)

    def run(n_rows):
        rows = np.sort(rng.choice(total_rows, size=n_rows, replace=False))
        b = (rows // w.L) // w.Hq
        i = rows % w.L
        flops = 4.0 * w.D * float(keys[b, i].sum())
        t0 = time.perf_counter()
        oracle.attn_fwd_f64(qd, kd, vd, w.sm_scale, causal=w.causal, valid_len=vln, rows=rows,
                            threads=threads)
        return time.perf_counter() - t0, flops, n_rows

    # calibrate on a small sample, then size the measured sample to the budget
    n = min(total_rows, 64 * max(1, oracle.max_threads()))
    dt, fl, _ = run(n)
    per_row = dt / n
    n_rows = int(min(total_rows, max(n, budget_s / max(per_row, 1e-9))))
    dt, fl, n_rows = run(n_rows)
    tflops = fl * ratio / dt / 1e12
    return tflops, {"rows": n_rows, "seconds": dt, "algorithmic_flops": fl,
                    "nominal_per_algorithmic": ratio}


# ------------------------------------------------------------------ GPU arm

def copies_only_ms(dev, host_in, host_out, reps=5):
    """The bytes of one end-to-end step moved with no kernel: every input host
    -> device on one stream while every output goes device -> host on another
    (the floor the pipelined host path approaches)."""
    import torch
    d_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in]
    d_out = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_out]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_out.wait_event(e0)
        with torch.cuda.stream(s_in):
            for d, h in zip(d_in, host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for d, h in zip(d_out, host_out):
                h.copy_(d, non_blocking=True)
        s_in.wait_stream(s_out)
        e1.record(s_in)
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    return best


def time_graph_loop(attn, w, x, dev, calls=1000, reps=5):
    """Per-call time of `calls` attn_fwd calls captured in one CUDA graph
    (inputs resident, no L2 flush: the whole problem of a launch-bound
    workload fits in L2).  x: the workload's Inputs."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        x.call(attn, side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream(dev)
        for _ in range(calls):
            x.call(attn, cap)
    g.replay()
    torch.cuda.synchronize(dev)
    best = float("inf")
    st = torch.cuda.current_stream(dev)
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.replay()
        e1.record(st)
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    status, code = attn.status(st)
    if status != 0:
        raise RuntimeError("device status after the graph loop: %d (code %#x)" % (status, code))
    del g
    us = best * 1e3 / calls
    return {"calls_per_graph": calls, "us_per_call": round(us, 3),
            "tflops": round(nominal_flops(w) / (us * 1e-6) / 1e12, 4),
            "timing": "CUDA events around one replay of the graph, best of %d" % reps}


O_ATOL, O_RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-4
PARITY_BOUND = "|o - o_ref| <= 2e-3 + 1e-2 |o_ref| per element; |lse - lse_ref| <= 1e-4, -inf matched"


def parity_summary(o, lse, o_ref, lse_ref) -> dict:
    """The GPU's O and LSE against the oracle's, every element: max abs and max
    rel error of O (rel over |o_ref| >= 1e-3), the worst error-to-bound ratio,
    the number of O elements over the bound, the LSE error and -inf pattern."""
    o = o.reshape(o_ref.shape)
    err = np.abs(o - o_ref)
    aref = np.abs(o_ref)
    bound = O_ATOL + O_RTOL * aref
    big = aref >= 1e-3
    lse = lse.reshape(lse_ref.shape)
    neg = np.isneginf(lse_ref)
    lerr = np.abs(lse[~neg] - lse_ref[~neg])
    n_over = int((err > bound).sum()) + int(np.sum(~np.isfinite(o)))
    n_lse_over = int((lerr > LSE_ATOL).sum()) + int((np.isneginf(lse) != neg).sum())
    return {
        "rows_compared": int(lse_ref.size),
        "max_abs_err_O": float(err.max()) if err.size else 0.0,
        "max_rel_err_O": float((err[big] / aref[big]).max()) if big.any() else 0.0,
        "worst_err_over_bound_O": round(float((err / bound).max()), 4) if err.size else 0.0,
        "max_err_LSE": float(lerr.max()) if lerr.size else 0.0,
        "n_over_bound": n_over + n_lse_over,
        "bound": PARITY_BOUND,
    }


def oracle_full(w, q, k, v, vl, threads: int = 0):
    """The float64 oracle over every row of the workload, timed: (o_ref, lse_ref,
    seconds).  This is the CPU-baseline leg; its outputs are also the parity
    reference."""
    import oracle
    t0 = time.perf_counter()
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(w.dtype),
                                          w.sm_scale, causal=w.causal,
                                          valid_len=None if vl is None else vl.numpy(),
                                          threads=threads)
    return o_ref, lse_ref, time.perf_counter() - t0


def time_calls(call, n, flush, stream):
    """Device ms of n calls, each bracketed by its own CUDA events on `stream`,
    with L2 flushed (a 256 MB write) before each, outside the events."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


class Inputs:
    """One workload's seeded inputs on the host and on the device, with outputs."""

    def __init__(self, w, dev, attn):
        self.w = w
        self.q, self.k, self.v, self.vl = wl.workload_inputs(w)
        self.q_d, self.k_d, self.v_d = self.q.to(dev), self.k.to(dev), self.v.to(dev)
        self.vl_d = None if self.vl is None else self.vl.to(dev)
        self.o_d = torch.empty_like(self.q_d)
        self.lse_d = torch.empty((w.B * w.Hq, w.L), dtype=torch.float32, device=dev)
        # the call's workspace (bf16: the fp16 copy of V), allocated once by torch
        n = attn.fwd_workspace_size(w.B, w.Hq, w.Hkv, w.L, w.L, w.D,
                                    attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev) if n else None

    def call(self, attn, stream):
        w = self.w
        attn.attn_fwd(self.q_d, self.k_d, self.v_d, causal=w.causal, sm_scale=w.sm_scale,
                      valid_len=self.vl_d, out=self.o_d, lse=self.lse_d, stream=stream,
                      workspace=self.ws)


def work_record(w, vl, ms_list, peaks):
    """Timing and roofline fractions of one workload from per-call device ms."""
    vln = None if vl is None else vl.numpy()
    nom = nominal_flops(w)
    alg = algorithmic_flops(w, vln)
    b = sum(io_bytes(w).values())
    med = statistics.median(ms_list)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = b / (med * 1e-3) / 1e9
    return {
        "workload": "%s: %s" % (w.name, w.description),
        "valid_len": None if vl is None else vl.tolist(),
        "calls_timed": len(ms_list),
        "ms_median": round(med, 5),
        "ms_p10": round(float(np.percentile(ms_list, 10)), 5),
        "ms_p90": round(float(np.percentile(ms_list, 90)), 5),
        "tflops_nominal": round(nom / (med * 1e-3) / 1e12, 3),
        "tflops_algorithmic": round(alg / (med * 1e-3) / 1e12, 3),
        "tensor_peak_frac_algorithmic": round(alg / (med * 1e-3) / 1e12 / peak, 4),
        "hbm_min_bytes": b,
        "hbm_gbs_at_min_bytes": round(gbs, 1),
        "hbm_peak_frac": round(gbs / hbm, 4),
        "nominal_flops": nom,
        "algorithmic_flops": alg,
    }


def run_gpu(args, w, world, rank, local):
    import attention_forward_attn_gb300 as attn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    attn.load()
    peaks, peak_src = load_peaks()
    x = Inputs(w, dev, attn)
    q, k, v, vl = x.q, x.k, x.v, x.vl
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        x.call(attn, stream)

    # calls per step: enough for ~args.step_ms of device time (estimated from
    # three calls after two untimed ones)
    for _ in range(2):
        flush.zero_()
        call()
    est = statistics.median(time_calls(call, 3, flush, stream))
    R = args.calls_per_step or int(max(1, min(2000, math.ceil(args.step_ms / max(est, 1e-3)))))
    for _ in range(args.warmup):
        for _ in range(R):
            flush.zero_()
            call()
    st, code = attn.status(stream)
    if st != 0:
        raise RuntimeError("device status after warm-up: %d (code %#x)" % (st, code))

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    wall0 = time.perf_counter()
    per_call = time_calls(call, args.steps * R, flush, stream)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    barrier(world)
    st, code = attn.status(stream)
    if st != 0:
        raise RuntimeError("device status after timing: %d (code %#x)" % (st, code))
    step_ms = [sum(per_call[s * R:(s + 1) * R]) for s in range(args.steps)]
    ms_mean = sum(step_ms) / len(step_ms)
    ms_max_rank = reduce_max(ms_mean, world)
    call_ms_mean = ms_mean / R

    # launch-bound workloads: the same call captured 1000 times in one CUDA
    # graph and replayed, so the per-call device time excludes launch latency
    graph_loop = None
    if call_ms_mean < 0.05:
        graph_loop = time_graph_loop(attn, w, x, dev)

    # end to end through the public API: attn_fwd_host takes the pinned host
    # buffers, copies the inputs in and the outputs back, pipelined with the kernels
    q_h, k_h, v_h = q.pin_memory(), k.pin_memory(), v.pin_memory()
    vl_h = None if vl is None else vl.pin_memory()
    o_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lse_h = torch.empty((w.B * w.Hq, w.L), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, args.e2e_steps)

    def e2e_step():
        attn.attn_fwd_host(q_h, k_h, v_h, causal=w.causal, sm_scale=w.sm_scale, valid_len=vl_h,
                           out=o_h, lse=lse_h, stream=stream, synchronize=False)

    e2e_chunks = attn.host_plan(w.B, w.Hq, w.Hkv, w.L, w.D,
                                attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    host_s = 0.0
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        e2e_step()
        host_s += time.perf_counter() - t0
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    st, code = attn.status(stream)
    if st != 0:
        raise RuntimeError("device status after e2e: %d (code %#x)" % (st, code))
    link_ms = copies_only_ms(dev, [q_h, k_h, v_h] + ([vl_h] if vl_h is not None else []),
                             [o_h, lse_h])
    del q_h, k_h, v_h, vl_h, o_h, lse_h

    # results
    vln = None if vl is None else vl.numpy()
    nom = nominal_flops(w)
    alg = algorithmic_flops(w, vln)
    # the timed region is seconds of back-to-back calls (the power cap can
    # act): the sustained peak is the denominator; the burst one is reported too
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = alg / (call_ms_mean * 1e-3) / 1e12
    b = io_bytes(w)
    launches_per_call = 2 if w.dtype == "bf16" else 1
    line = {
        "metric": METRIC,
        "value": round(aggregate(nom * R, ms_max_rank * 1e-3, world), 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max_rank, 5),
        "ms_per_call": round(ms_max_rank / R, 5),
        "calls_per_step": R,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) fp32 rounded to %s%s" % (
            w.dtype, ", Q x%g" % w.q_scale if w.q_scale != 1.0 else ""),
        "config": {
            "workload": "%s: %s" % (w.name, w.description),
            "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L, "D": w.D, "causal": w.causal,
            "valid_len": None if vl is None else vl.tolist(), "sm_scale": w.sm_scale,
            "parallelism": "replicas x%d (no exchange step)" % world,
            "l2": "flushed before every timed call (256 MB write, outside the events)",
            "timing": ("a step = %d attn_fwd calls, each bracketed by CUDA events on its stream "
                       "(%s); the step's time is the sum of its calls' times" % (
                           R, "bf16: V pre-pass + attention kernel" if w.dtype == "bf16"
                           else "attention kernel")),
            "ms_per_call_median": round(statistics.median(per_call), 5),
            "ms_per_call_p10": round(float(np.percentile(per_call, 10)), 5),
            "ms_per_call_p90": round(float(np.percentile(per_call, 90)), 5),
            "wall_s_timed_region": round(wall, 4),
            "nominal_flops_per_call": nom,
            "algorithmic_flops_per_call": alg,
        },
        "roofline": {
            "bound": "tensor",
            "achieved": round(achieved, 3),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_source": ("%s bf16_tflops_sustained (the timed region is %.1f s of back-to-back "
                            "calls)" % (peak_src, wall)),
            "peak_burst": peak_burst,
            "frac_of_burst_peak": round(achieved / peak_burst, 4),
            "traffic": committed_traffic(w.name),
            "traffic_unit": "bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)",
            "hbm_min_bytes": sum(b.values()),
            "hbm_gbs_at_min_bytes": round(sum(b.values()) / (call_ms_mean * 1e-3) / 1e9, 1),
            "hbm_peak_gbs": float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
        },
        "e2e": {
            "value": round(aggregate(nom, e2e_ms * 1e-3, world), 3),
            "unit": UNIT,
            "h2d_bytes_per_step": b["q"] + b["kv"] + b["valid_len"],
            "d2h_bytes_per_step": b["o"] + b["lse"],
            "ms_per_step": round(e2e_ms, 4),
            "steps": e2e_steps,
            "path": ("attn_fwd_host (C ABI via the binding): pinned host Q/K/V/O/LSE, "
                     "copies pipelined with the kernels in %d chunks; one call per step" % len(
                         e2e_chunks)),
            "copies_only_ms_per_step": round(link_ms, 4),
            "host_queue_ms_per_step": round(host_s * 1e3 / e2e_steps, 4),
        },
        # attn_fwd launches the attention kernel, preceded for bf16 by the
        # kernel that makes the fp16 copy of V
        "gpu_launches": args.steps * R * launches_per_call,
        "graph_loop": graph_loop,
        "clocks": clocks,
    }
    if rank != 0 or args.no_cpu_baseline:
        return line

    # The CPU-baseline leg: the float64 oracle over the whole workload, timed
    # on the host cores; its outputs are the parity reference for the GPU's.
    # First the headline workload, then (unless --no-workloads) every other one.
    call()
    torch.cuda.synchronize(dev)
    o_gpu = x.o_d.float().cpu().numpy()
    lse_gpu = x.lse_d.cpu().numpy()
    threads = _oracle_threads()
    o_ref, lse_ref, secs = oracle_full(w, q, k, v, vl)
    line["parity"] = dict(workload=w.name, **parity_summary(o_gpu, lse_gpu, o_ref, lse_ref))
    del o_gpu, lse_gpu, o_ref, lse_ref
    line["cpu_baseline"] = {
        "value": round(nom / secs / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
        "sample": "the whole workload: all %d query rows of %s (%.1f s of float64 oracle work)" % (
            w.B * w.Hq * w.L, w.name, secs),
        "single_thread": single_thread_times(),
    }
    headline = work_record(w, vl, per_call, peaks)
    headline["parity"] = line["parity"]
    headline["cpu_oracle_s"] = round(secs, 2)
    if graph_loop is not None:
        headline["graph_loop"] = graph_loop
    del x
    torch.cuda.empty_cache()
    if args.no_workloads:
        return line
    recs = {}
    for name in sorted(wl.WORKLOADS):
        if name == w.name:
            recs[name] = headline
            continue
        wk = wl.WORKLOADS[name]
        y = Inputs(wk, dev, attn)

        def call_y():
            y.call(attn, stream)

        for _ in range(10):  # warm-up calls
            flush.zero_()
            call_y()
        ms = time_calls(call_y, args.workload_calls, flush, stream)
        st, code = attn.status(stream)
        if st != 0:
            raise RuntimeError("device status on %s: %d (code %#x)" % (name, st, code))
        rec = work_record(wk, y.vl, ms, peaks)
        if statistics.median(ms) < 0.05:
            rec["graph_loop"] = time_graph_loop(attn, wk, y, dev)
        call_y()
        torch.cuda.synchronize(dev)
        o_gpu = y.o_d.float().cpu().numpy()
        lse_gpu = y.lse_d.cpu().numpy()
        o_ref, lse_ref, secs = oracle_full(wk, y.q, y.k, y.v, y.vl)
        rec["parity"] = parity_summary(o_gpu, lse_gpu, o_ref, lse_ref)
        rec["cpu_oracle_s"] = round(secs, 2)
        recs[name] = rec
        del y, o_gpu, lse_gpu, o_ref, lse_ref
        torch.cuda.empty_cache()
    line["workloads"] = recs
    line["workloads_note"] = (
        "per workload: 10 warm-up and %d timed calls (the headline: the timed steps' calls), L2 "
        "flushed before each, "
        "CUDA events; fractions of the %s peaks (bf16_tflops burst, hbm_gbs) from algorithmic "
        "FLOPs and the minimum bytes Q+K+V+O+LSE; parity: the whole output against the float64 "
        "oracle run over the whole workload on %d host cores (cpu_oracle_s)" % (
            args.workload_calls, peak_src, threads))
    return line


def single_thread_times():
    """The oracle on one host thread: C1 whole, and C2 on a random sample of
    query rows of about 5 s (scaled to the whole workload)."""
    out = {}
    w1 = wl.WORKLOADS["C1"]
    q, k, v, vl = wl.workload_inputs(w1)
    _, _, secs = oracle_full(w1, q, k, v, vl, threads=1)
    out["C1"] = {"seconds": round(secs, 4), "tflops": round(nominal_flops(w1) / secs / 1e12, 6),
                 "rows": "all %d" % (w1.B * w1.Hq * w1.L)}
    w2 = wl.WORKLOADS["C2"]
    q, k, v, vl = wl.workload_inputs(w2)
    tfl, det = oracle_sample(w2, q, k, v, vl, 5.0, np.random.default_rng(4321), threads=1)
    out["C2"] = {"seconds": round(det["seconds"], 3), "tflops": round(tfl, 6),
                 "rows": "%d random of %d" % (det["rows"], w2.B * w2.Hq * w2.L),
                 "seconds_whole_workload_extrapolated": round(nominal_flops(w2) / (tfl * 1e12), 1)}
    return out


def mask_workloads(dev):
    """The explicit-mask workloads: (name, workload, keep-mask builder, implicit
    kwargs or None).  The builders return a bool [B or 1, L, L] device tensor."""
    def padding(w, vl_d):
        L = w.L
        return torch.arange(L, device=dev)[None, None, :] < vl_d[:, None, None].expand(w.B, L, 1)

    def tril(w, vl_d):
        return torch.tril(torch.ones(w.L, w.L, dtype=torch.bool, device=dev))[None]

    def band(w, vl_d):
        i = torch.arange(w.L, device=dev)[:, None]
        j = torch.arange(w.L, device=dev)[None, :]
        return (((i - j).abs() < 512) | (j < 256))[None]

    return [
        ("C3 padding as an explicit [8,4096,4096] mask", wl.WORKLOADS["C3"], padding,
         dict(causal=False, padded=True)),
        ("C4 causal as an explicit tril [4096,4096] mask", wl.WORKLOADS["C4"], tril,
         dict(causal=True, padded=False)),
        ("C4 shapes, causal, band |i-j| < 512 plus keys < 256", wl.WORKLOADS["C4"], band, None),
    ]


def run_mask_workloads(args, local):
    """One JSON line per explicit-mask workload: ms per attn_fwd_masked call
    (mask pre-pass + bf16 V pre-pass + attention, L2 flushed before each call)
    and, where the mask restates an implicit one, the implicit call's ms."""
    import attention_forward_attn_gb300 as attn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    attn.load()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks, peak_src = load_peaks()
    lines = []
    for name, w, build, implicit in mask_workloads(dev):
        q, k, v, vl = wl.workload_inputs(w)
        q_d, k_d, v_d = q.to(dev), k.to(dev), v.to(dev)
        vl_d = None if vl is None else vl.to(dev)
        keep = build(w, vl_d)
        causal_masked = implicit is None and w.causal
        o_d = torch.empty_like(q_d)
        lse_d = torch.empty((w.B * w.Hq, w.L), dtype=torch.float32, device=dev)

        def timed(fn, n):
            for _ in range(args.warmup):
                flush.zero_()
                fn()
            ts = []
            for _ in range(n):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            st, code = attn.status()
            if st != 0:
                raise RuntimeError("device status %d (code %#x)" % (st, code))
            return sorted(ts)[len(ts) // 2]

        n = max(5, min(args.steps, 200))
        ms_mask = timed(lambda: attn.attn_fwd_strided(q_d, k_d, v_d, causal=causal_masked,
                                                      sm_scale=w.sm_scale, mask=keep, out=o_d,
                                                      lse=lse_d), n)
        ms_impl = None
        if implicit is not None:
            ms_impl = timed(lambda: attn.attn_fwd(q_d, k_d, v_d, causal=implicit["causal"],
                                                  sm_scale=w.sm_scale,
                                                  valid_len=vl_d if implicit["padded"] else None,
                                                  out=o_d, lse=lse_d), n)
        # visible (query, key) pairs of every head: the algorithmic work
        vis = keep.expand(w.B, w.L, w.L)
        if causal_masked:
            vis = vis & torch.tril(torch.ones(w.L, w.L, dtype=torch.bool, device=dev))
        pairs = float(vis.sum().item()) * w.Hq
        flops = 4.0 * w.D * pairs
        tf = flops / (ms_mask * 1e-3) / 1e12
        lines.append({
            "metric": "attention fwd TFLOP/s with an explicit boolean mask (algorithmic)",
            "workload": name, "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_call": round(ms_mask, 4),
            "implicit_ms_per_call": None if ms_impl is None else round(ms_impl, 4),
            "visible_pairs_per_head_all_batches": int(pairs / w.Hq),
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                         "peak_source": "%s bf16_tflops" % peak_src},
            "timing": "median of %d calls, L2 flushed before each, CUDA events; the call includes "
                      "the mask pre-pass and the bf16 V pre-pass" % n,
            "dtype": w.dtype, "data": "synthetic"})
        del keep, q_d, k_d, v_d, o_d, lse_d
        torch.cuda.empty_cache()
    return lines


def run_relative_table(args, local):
    """The comparison of "masked multi head attention in CUDA" section 6.1,
    on this GPU: B=1, H=8, N=1024, D=64, fp32, causal mask, rows = the
    unfused PyTorch path (scores, mask, softmax, then V; TF32 off, as the
    page's section 5.3 asks), the naive three-pass kernel, the tiled kernel
    with a per-element online softmax, the tiled kernel with the block row
    max (the page's 1.0x), and the tcgen05 kernel on bf16 / fp16 copies of
    the inputs.  Times: median of the timed calls, L2 flushed before each."""
    import attention_forward_attn_gb300 as attn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    attn.load()
    B, H, L, D = 1, 8, 1024, 64
    gen = torch.Generator().manual_seed(26)
    q, k, v = (torch.randn(B, H, L, D, generator=gen).to(dev) for _ in range(3))
    sm = 1.0 / D ** 0.5
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    keep = torch.tril(torch.ones(L, L, dtype=torch.bool, device=dev))
    old_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False

    def torch_unfused():
        s_ = torch.matmul(q, k.transpose(-1, -2)) * sm
        s_ = s_.masked_fill(~keep, float("-inf"))
        return torch.matmul(torch.softmax(s_, dim=-1), v)

    qb, kb, vb = q.bfloat16(), k.bfloat16(), v.bfloat16()
    qh, kh, vh = q.half(), k.half(), v.half()
    impls = [
        ("PyTorch unfused (scores, mask, softmax, V), fp32", torch_unfused, 4.0),
        ("naive CUDA kernel (three passes), fp32",
         lambda: attn.attn_fwd_f32(q, k, v, kernel="naive", causal=True, sm_scale=sm), 3.2),
        ("tiled CUDA kernel, per-element online softmax, fp32",
         lambda: attn.attn_fwd_f32(q, k, v, kernel="tiled_element", causal=True, sm_scale=sm), 1.4),
        ("tiled CUDA kernel, block row max, fp32",
         lambda: attn.attn_fwd_f32(q, k, v, kernel="tiled_rowmax", causal=True, sm_scale=sm), 1.0),
        ("tcgen05 kernel (attn_fwd), bf16 inputs",
         lambda: attn.attn_fwd(qb, kb, vb, causal=True, sm_scale=sm), None),
        ("tcgen05 kernel (attn_fwd), fp16 inputs",
         lambda: attn.attn_fwd(qh, kh, vh, causal=True, sm_scale=sm), None),
    ]
    rows = []
    n = max(5, min(args.steps, 100))
    for name, fn, page in impls:
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        fn()
        torch.cuda.synchronize(dev)
        extra = torch.cuda.max_memory_allocated(dev) - base
        ts = []
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        st, code = attn.status()
        if st != 0:
            raise RuntimeError("device status %d (code %#x)" % (st, code))
        rows.append({"impl": name, "ms": round(sorted(ts)[n // 2], 4), "page_relative": page,
                     "torch_peak_extra_bytes": int(extra)})
    torch.backends.cuda.matmul.allow_tf32 = old_tf32
    ref = [r for r in rows if r["page_relative"] == 1.0][0]["ms"]
    for r in rows:
        r["relative_to_tiled_rowmax"] = round(r["ms"] / ref, 3)
    return {"metric": "relative time of attention implementations (masked multi head attention "
                      "in CUDA, section 6.1), B=1 H=8 N=1024 D=64 causal",
            "rows": rows, "timing": "median of %d calls, L2 flushed before each, CUDA events" % n,
            "note": "page_relative: the page's own factors (one Ampere GPU, single runs); "
                    "torch_peak_extra_bytes: device memory torch allocated during one call "
                    "(the fused kernels allocate none through torch)",
            "data": "synthetic N(0,1), seed 26"}


def run_backward(args, local):
    """attn_bwd (tensor cores) and attn_bwd_simt (fp32 SIMT) on the C4, C2 and
    C5 shapes, and attn_bwd_masked on C4M -- C4 with its causal mask given as
    an explicit tril mask -- (--bwd-workloads): ms per call with the forward's O and LSE already on the device,
    L2 flushed before each call.  Work: the backward's five products (S
    recomputed, dP, dQ, dK, dV) = 2.5x the forward's nominal FLOPs.  The
    tensor-core path executes seven (S and dP in both of its kernels), 3.5x.
    Rooflines: tensor -- the measured bf16 burst peak (fp16 runs at the same
    rate), against the executed products; SIMT -- the FP32 units, 152 SMs x
    128 FMA lanes x 2 FLOP x the 2070 MHz maximum SM clock = 80.6 TFLOP/s."""
    import attention_forward_attn_gb300 as attn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    attn.load()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks, src = load_peaks()
    fp32_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    tc_peak = peaks["bf16_tflops"]
    lines = []
    impls = ("tc", "simt") if args.bwd_impl == "both" else (args.bwd_impl,)
    for name in args.bwd_workloads.split(","):
        # "C4M": C4's shapes with its causal mask given as an explicit boolean
        # [L, L] mask (attn_bwd_masked; every tile computed, none skipped)
        masked = name.endswith("M")
        w = wl.WORKLOADS[name[:-1] if masked else name]
        q, k, v, vl = wl.workload_inputs(w)
        q_d, k_d, v_d = q.to(dev), k.to(dev), v.to(dev)
        vl_d = None if vl is None else vl.to(dev)
        gen = torch.Generator().manual_seed(w.seed + 100)
        do = torch.randn(q.shape, generator=gen).to(q.dtype).to(dev)
        o, lse = attn.attn_fwd(q_d, k_d, v_d, causal=w.causal, sm_scale=w.sm_scale, valid_len=vl_d)
        mk = torch.tril(torch.ones(w.L, w.L, dtype=torch.bool, device=dev)) if masked else None
        for impl in (("tc",) if masked else impls):
            def call():
                return attn.attn_bwd(q_d, k_d, v_d, o, lse, do, causal=w.causal and not masked,
                                     sm_scale=w.sm_scale, valid_len=vl_d, impl=impl, mask=mk)

            for _ in range(max(1, min(args.warmup, 3))):
                flush.zero_()
                call()
            n = max(3, min(args.steps, 10 if impl == "simt" else 50))
            ts = []
            for _ in range(n):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            st, code = attn.status()
            if st != 0:
                raise RuntimeError("device status %d (code %#x)" % (st, code))
            ms = sorted(ts)[n // 2]
            tf = 2.5 * nominal_flops(w) / (ms * 1e-3) / 1e12
            if impl == "tc":
                ex = 3.5 * nominal_flops(w) / (ms * 1e-3) / 1e12
                roof = {"bound": "tensor", "achieved": round(ex, 3), "peak": tc_peak,
                        "unit": "TFLOP/s", "frac": round(ex / tc_peak, 4),
                        "peak_source": "bf16_tflops of %s (burst), executed products (3.5x)" % src}
            else:
                roof = {"bound": "alu", "achieved": round(tf, 3), "peak": round(fp32_peak, 1),
                        "unit": "TFLOP/s", "frac": round(tf / fp32_peak, 4),
                        "peak_source": "152 SMs x 128 FP32 lanes x 2 x sm_max_mhz"}
            lines.append({"metric": "attention backward TFLOP/s (2.5x the forward's nominal FLOPs)",
                          "impl": ("attn_bwd_masked" if masked else "attn_bwd") if impl == "tc"
                          else "attn_bwd_simt",
                          "workload": "%s shapes: %s%s" % (name, w.description,
                                                           ", as an explicit tril mask" if masked else ""),
                          "value": round(tf, 3),
                          "unit": "TFLOP/s", "ms_per_call": round(ms, 3), "roofline": roof,
                          "timing": "median of %d calls, L2 flushed before each" % n,
                          "dtype": w.dtype, "data": "synthetic"})
        del q_d, k_d, v_d, o, lse, do
        torch.cuda.empty_cache()
    return lines


def _oracle_threads() -> int:
    import oracle
    return oracle.max_threads()


# ------------------------------------------------------------------ reference arm

def run_reference(args, w):
    """The float64 CPU oracle as the reference arm: each step a bounded random
    sample of the workload's query rows.  value: the sampled rows' work (in the
    metric's nominal-FLOP convention) over the time they took; ms_per_step: the
    measured time of a step's sample."""
    q, k, v, vl = wl.workload_inputs(w)
    rng = np.random.default_rng(99)
    per_step = max(0.2, args.reference_budget_s / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, vl, per_step, rng)
    flops, secs, rows = 0.0, [], 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tfl, det = oracle_sample(w, q, k, v, vl, per_step, rng)
        flops += tfl * 1e12 * det["seconds"]
        secs.append(det["seconds"])
        rows += det["rows"]
    wall = time.perf_counter() - t0
    value = flops / sum(secs) / 1e12
    nom = nominal_flops(w)
    cores = _oracle_threads()
    ms_step = sum(secs) / len(secs) * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded N(0,1) rounded to %s, decoded to float64" % w.dtype,
        "config": {"workload": "%s: %s" % (w.name, w.description), "B": w.B, "Hq": w.Hq,
                   "Hkv": w.Hkv, "L": w.L, "D": w.D, "causal": w.causal,
                   "step": "a random sample of %d query rows on average (of %d)" % (
                       rows // max(1, args.steps), w.B * w.Hq * w.L),
                   "ms_whole_workload_extrapolated": round(nom / (value * 1e12) * 1e3, 1),
                   "wall_s_timed_steps": round(wall, 2)},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": "%d random query rows per step on average (%.2f s each)" % (
                             rows // max(1, args.steps), sum(secs) / len(secs))},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="C4", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle leg (CPU baseline and parity)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="only the headline workload (no per-workload record)")
    ap.add_argument("--calls-per-step", type=int, default=0,
                    help="attn_fwd calls per timed step (0: enough for --step-ms)")
    ap.add_argument("--step-ms", type=float, default=120.0,
                    help="device time a timed step aims at when --calls-per-step is 0")
    ap.add_argument("--workload-calls", type=int, default=50,
                    help="timed calls per workload of the per-workload record")
    ap.add_argument("--mask-workloads", action="store_true",
                    help="instead of the headline line, one line per explicit-mask workload")
    ap.add_argument("--relative-table", action="store_true",
                    help="instead of the headline line, the section 6.1 comparison table")
    ap.add_argument("--backward", action="store_true",
                    help="instead of the headline line, one line per backward workload")
    ap.add_argument("--bwd-impl", default="both", choices=["both", "tc", "simt"],
                    help="--backward: which backward (attn_bwd, attn_bwd_simt or both)")
    ap.add_argument("--bwd-workloads", default=BWD_WORKLOADS,
                    help="--backward: comma-separated workload shapes")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.WORKLOADS[args.workload]
    world, rank, local = dist_env()
    if world != args.gpus and world > 1:
        ap.error("--gpus %d does not match WORLD_SIZE %d" % (args.gpus, world))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return 0
    if args.backward:
        if rank == 0:
            for line in run_backward(args, local):
                print(json.dumps(line), flush=True)
        return 0
    if args.relative_table:
        if rank == 0:
            print(json.dumps(run_relative_table(args, local)), flush=True)
        return 0
    if args.mask_workloads:
        if rank == 0:
            for line in run_mask_workloads(args, local):
                print(json.dumps(line), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    line = run_gpu(args, w, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
