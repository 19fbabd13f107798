#!/usr/bin/env python3
"""Benchmark of the fused conv + norm forward on GB300.

Default workload: Conv3d(3->16, k=4) on (512, 3, 16, 32, 32) -> HardSwish ->
GroupNorm(4) -> mean over D,H,W (the conv tensor is never materialised).
A step is one conv_norm_forward over the whole batch, inputs resident in
HBM; L2 is flushed (256 MB write) before every timed step because the input
(100 MB) fits in L2.  The metric is GFLOP/s of algorithmic conv FLOPs
(2 per multiply-add over the outputs the method must compute) with the
time per step; the roofline is max(FLOPs / FP32 peak, compulsory bytes /
HBM bandwidth).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference] [--no-extras] [--no-cpu-baseline] [--batch N]

Under torchrun each rank runs its own full batch (weak scaling, no
collective on the data path); the value is the sum of FLOPs over ranks
divided by the slowest rank's time.  --impl reference times the fp64 CPU
oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from convolution_normalization_gb300 import workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "conv3d_hswish_gn4_mean_n512"
# SM count when no device is visible (host-only runs); the CUDA arm reads the
# device's own count
DEFAULT_SMS = 152
FP32_LANES_PER_SM = 128
METRIC = "fused conv+norm forward ms & GFLOP/s, % of roofline (FP32 peak vs HBM)"
DATA = "synthetic (seeded PCG64: x~N(0,1), w,b~U(+-1/sqrt(fan_in)), gamma=1+0.1N, beta=0.1N)"


# ---- workload arithmetic (for reporting only) ---------------------------------

def conv_out_dims(s):
    k = s["k"]
    if s["conv"] == "conv3d":
        return [s["D"] - k + 1, s["H"] - k + 1, s["W"] - k + 1]
    if s["conv"] == "conv2d":
        return [s["H"] - k + 1, s["W"] - k + 1]
    return [s["H"] + k - 1, s["W"] + k - 1]


def algorithmic_flops(s):
    """2 x multiply-adds over the conv outputs the method must compute (for
    the double max-pool only the kept 4*floor(L/4) region)."""
    dims = conv_out_dims(s)
    if s["red"] == "maxpool2_x2":
        dims = [4 * (L // 4) for L in dims]
    taps = (s["C_in"] // s["groups"]) * s["k"] ** (3 if s["conv"] == "conv3d" else 2)
    return 2.0 * s["N"] * s["C_out"] * math.prod(dims) * taps


def out_shape(s):
    dims = conv_out_dims(s)
    if s["red"] == "mean_spatial":
        return (s["N"], s["C_out"])
    if s["red"] == "maxpool2_x2":
        return (s["N"], s["C_out"], *[(L // 2) // 2 for L in dims])
    return (s["N"], s["C_out"], *dims)


def compulsory_bytes(s):
    shp = wl.input_shapes(s)
    n = sum(math.prod(v) for v in shp.values() if v)
    return 4.0 * (n + math.prod(out_shape(s)))


def peaks(sms=None):
    """Roofline denominators: measured HBM copy bandwidth and bf16 GEMM rate
    (MEASURED_PEAKS.json, else the stated fallback) and the FP32 FMA peak
    from the SM count (the device's, when given), 128 FP32 lanes per SM and
    the maximum SM clock."""
    p = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
    hbm = p.get("hbm_gbs")
    sm_mhz = p.get("sm_max_mhz") or 2070.0
    src = "measured" if hbm else "fallback"
    if not hbm:
        hbm = 6800.0
    sms_src = "device" if sms else "default"
    sms = sms or DEFAULT_SMS
    fp32 = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12  # TFLOP/s
    bf16 = p.get("bf16_tflops") or 1900.0
    return dict(hbm_gbs=hbm, fp32_tflops=fp32, sm_max_mhz=sm_mhz, source=src, bf16_tflops=bf16,
                sms=sms, sms_source=sms_src)


def roofline_ms(s, pk):
    t_c = algorithmic_flops(s) / (pk["fp32_tflops"] * 1e12)
    t_m = compulsory_bytes(s) / (pk["hbm_gbs"] * 1e9)
    return 1e3 * max(t_c, t_m), ("alu" if t_c >= t_m else "hbm")


# ---- ncu traffic figure (only while the kernel source is unchanged) ------------

_CS = "convolution_normalization_gb300/csrc/"
# the source files each kernel is built from (its profile is current while
# their hash is unchanged)
KERNEL_SOURCES = {
    "k_conv3d_act_mean": ("k_conv3d_mean.cu", "cn_mean_common.cuh", "cn_common.cuh"),
    "k_conv3d_softmax_pool4": ("k_conv3d_softmax_pool.cu", "cn_common.cuh"),
    "k_conv2d_act_stats": ("k_conv2d_norm.cu", "cn_common.cuh"),
    "k_conv2d_tc": ("k_conv2d_tc.cu", "cn_tcgen05.cuh", "cn_common.cuh"),
    "k_norm_apply": ("k_conv2d_norm.cu", "cn_common.cuh"),
    "k_conv3d_tc_mean": ("k_conv3d_tc.cu", "cn_tcgen05.cuh", "cn_common.cuh"),
    "k_conv3d_tc_pool": ("k_conv3d_tc.cu", "cn_tcgen05.cuh", "cn_common.cuh"),
    "k_convt2d_tc": ("k_convt2d_tc.cu", "cn_tcgen05.cuh", "cn_common.cuh"),
    "k_conv3d_mean_small": ("k_conv3d_mean_small.cu", "cn_common.cuh"),
}
# tf32 tensor peak from the measured bf16 one and the nominal dense ratio
# (1.1 / 2.25 PFLOP/s); split-TF32 runs 3 tf32 products per fp32 product
TF32_PER_BF16 = 1.1 / 2.25
SPLIT_TF32_PRODUCTS = 3
TC_KERNELS = ("k_conv2d_tc", "k_conv3d_tc_mean", "k_conv3d_tc_pool", "k_convt2d_tc")


def contraction(kernel_names):
    """The arithmetic of the conv of a plan's kernel list."""
    if any(k in kernel_names for k in TC_KERNELS):
        return "3xTF32 split on tcgen05 tensor cores, fp32 accumulate (fp32 accuracy)"
    return "fp32 FFMA on CUDA cores"


def split_names(s):
    """Kernel names of plan_info, split at the commas outside template < >."""
    out, depth, cur = [], 0, ""
    for ch in s:
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        if ch == "," and depth == 0:
            out.append(cur)
            cur = ""
        else:
            cur += ch
    if cur:
        out.append(cur)
    return out


def kernel_key(name):
    base = name.split("<")[0]
    return base if base in KERNEL_SOURCES else None


def source_hash(key):
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[key]:
        h.update(open(os.path.join(ROOT, _CS + p), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, key):
    """dram bytes per launch of the dominant kernel from
    profiles/<workload>.txt if it was captured from the current kernel source
    (its 'kernel' and 'source_hash' lines match)."""
    path = os.path.join(ROOT, "profiles", f"{workload}.txt")
    if key is None or not os.path.exists(path):
        return None
    txt = open(path).read()
    k = re.search(r"^kernel:\s*(\S+)", txt, re.M)
    m = re.search(r"^source_hash:\s*(\S+)", txt, re.M)
    t = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", txt, re.M)
    if not k or not m or not t or kernel_key(k.group(1)) != key or m.group(1) != source_hash(key):
        return None
    return float(t.group(1))


def kernel_roofline(spec, name, ms, pk):
    """Roofline of one kernel launch of the forward: the method's algorithmic
    work per launch / its measured duration, against the peak of the unit the
    kernel runs on (tf32 tensor pipe, HBM, or the FP32 pipe)."""
    flops = algorithmic_flops(spec)
    base = name.split("<")[0]
    if base in TC_KERNELS:
        ach = flops / (ms / 1e3) / 1e12
        peak = pk["bf16_tflops"] * TF32_PER_BF16
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "work": f"2 x MACs = {flops:.4g} flop (the method's own work)",
                "peak_source": f"measured bf16 {pk['bf16_tflops']} TFLOP/s x nominal tf32/bf16 "
                               f"{TF32_PER_BF16:.3f}",
                # what the tensor pipe executes: the split's 3 tf32 products per MAC
                "split_tf32": {"achieved": SPLIT_TF32_PRODUCTS * ach,
                               "frac": SPLIT_TF32_PRODUCTS * ach / peak,
                               "work": f"{SPLIT_TF32_PRODUCTS} tf32 products x 2 x MACs"},
                "frac_of_fp32_peak": ach / pk["fp32_tflops"]}
    if base == "k_norm_apply":
        nbytes = 2.0 * 4 * math.prod(out_shape(spec))
        return {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "work": f"read + write of the output = {nbytes:.4g} B",
                "peak_source": f"{pk['source']} HBM {pk['hbm_gbs']} GB/s"}
    return {"bound": "alu", "achieved": flops / (ms / 1e3) / 1e12, "peak": pk["fp32_tflops"],
            "unit": "TFLOP/s", "work": f"2 x MACs = {flops:.4g} flop",
            "peak_source": f"FP32: {pk['sms']} SMs ({pk['sms_source']}) x {FP32_LANES_PER_SM} "
                           f"lanes x 2 x {pk['sm_max_mhz']:.0f} MHz"}


def config_of(spec):
    """The workload a line is measured on: the same keys and values in both
    arms (the arithmetic each arm uses is its own top-level key)."""
    return {"workload": spec["name"], "N": spec["N"], "C_in": spec["C_in"],
            "C_out": spec["C_out"], "D": spec["D"], "H": spec["H"], "W": spec["W"],
            "k": spec["k"], "groups": spec["groups"], "per_rank_batch": spec["N"],
            "l2": "flushed before every timed GPU step (256 MB write)",
            "precision": "fp32 result, |err| <= 1e-4 + 1e-4|ref| against the fp64 oracle"}


# ---- clocks ----------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                pw.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        busy = [s for s, p in zip(sm, pw) if p > 0.3 * max(pw)] if pw else []
        return {"sm_mhz": statistics.median(busy or sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ---- distributed plumbing ----------------------------------------------------------

def dist_setup(n_gpus):
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE): NCCL
    with GPUs, gloo without (the host-side logic is tested that way)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    """The slowest rank's time: the job finishes when every rank has."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms_max):
    """Whole-job throughput: every rank processes its own batch (weak
    scaling, no data-path collective), the job takes the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


# ---- oracle (CPU baseline and the reference arm) --------------------------------------

def oracle_rate(spec, inp, target_s, max_samples=None):
    """Times the fp64 oracle on a bounded number of samples; returns
    (GFLOP/s, samples, seconds, threads)."""
    import oracle
    probe = min(spec["N"], 2)
    t0 = time.perf_counter()
    oracle.forward(spec, inp, samples=list(range(probe)))
    per = max((time.perf_counter() - t0) / probe, 1e-6)
    n = int(max(1, min(spec["N"], max_samples or spec["N"], target_s / per)))
    t0 = time.perf_counter()
    oracle.forward(spec, inp, samples=list(range(n)))
    dt = time.perf_counter() - t0
    flops = algorithmic_flops(wl.with_overrides(spec, N=n))
    return flops / dt / 1e9, n, dt, oracle.num_threads()


def run_reference(args, spec):
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = wl.make_inputs(spec)
    budget = 150.0 / max(1, args.steps + args.warmup)
    _, n, _, threads = oracle_rate(spec, inp, target_s=min(budget, 2.0))
    sub = list(range(n))
    for _ in range(args.warmup):
        oracle.forward(spec, inp, samples=sub)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(spec, inp, samples=sub)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    flops = algorithmic_flops(wl.with_overrides(spec, N=n))
    val = flops / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": config_of(spec),
        "contraction": "fp64 loops on the host cores (the oracle)",
        "cpu_baseline": {"value": val, "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} of {spec['N']} samples per step"},
        "e2e": {"value": val, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the CUDA path ------------------------------------------------------------------------

def time_forward(B, torch, plan, dev, out, stream, steps, warmup, flush_buf, nlaunch):
    """Times `steps` forwards (L2 flushed before each) with CUDA events on the
    forward's stream: the plan records one event before each kernel launch and
    one after the last, so a step is the time from its first event to its last
    (no events of its own beside them).  Returns (step ms list, per-launch ms
    lists)."""
    def fwd():
        plan.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], out, stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush_buf.zero_()
            fwd()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    lev = [[torch.cuda.Event(enable_timing=True) for _ in range(nlaunch + 1)]
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for row in lev:  # the CUDA events exist once recorded
            for e in row:
                e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        # Hold the stream for a moment so the host queues every step before
        # the device starts them: the per-step events then time the kernels,
        # not host enqueue latency.
        torch.cuda._sleep(int(min(2e9, 2e5 * steps + 2e7)))
        for i in range(steps):
            flush_buf.zero_()
            if nlaunch:
                plan.set_launch_events(lev[i])
                fwd()
            else:  # an empty problem launches nothing
                starts[i].record(stream)
                fwd()
                ends[i].record(stream)
    stream.synchronize()
    plan.set_launch_events(None)
    if nlaunch:
        step_ms = [row[0].elapsed_time(row[-1]) for row in lev]
    else:
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    launch_ms = [[lev[i][j].elapsed_time(lev[i][j + 1]) for i in range(steps)]
                 for j in range(nlaunch)]
    return step_ms, launch_ms


def measure(B, torch, spec, pk, stream, flush, steps, warmup, world=1, e2e_steps=10,
            cpu_target_s=None, sampler=None):
    """One workload on this rank: device step time (mean of `steps`, L2
    flushed before each), per-launch times, the dominant kernel's roofline,
    the step roofline of the workload's metric, the end-to-end time through
    the host-buffer entry point and (if cpu_target_s) the oracle's rate on
    the host cores."""
    inp = wl.make_inputs(spec)
    dev = {k: (torch.from_numpy(v).cuda() if v is not None else None) for k, v in inp.items()}
    plan = B.Plan(spec)
    info = plan.info()
    nl = info["launches_per_forward"]
    out = torch.empty(plan.out_shape, dtype=torch.float32, device="cuda")
    if sampler:
        barrier(world)
        torch.cuda.synchronize()
        sampler.start()
    times, launch_ms = time_forward(B, torch, plan, dev, out, stream, steps, warmup, flush, nl)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    assert plan.check_device(stream) == B.CN_OK
    ms_rank = statistics.mean(times)
    ms = max_over_ranks(world, ms_rank)
    flops = algorithmic_flops(spec)
    rl_ms, bound = roofline_ms(spec, pk)
    names = split_names(info["kernel_names"])[:nl]
    means = [statistics.mean(v) for v in launch_ms]
    dom = max(range(nl), key=lambda j: means[j])
    roofline = kernel_roofline(spec, names[dom], means[dom], pk)
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    roofline.update({
        "traffic": profiled_traffic(spec["name"], kernel_key(names[dom])),
        "kernel": names[dom], "kernel_ms": means[dom],
        "launch_ms": {n: m for n, m in zip(names, means)},
        # the workload's metric: FP32-peak / HBM roofline time of the whole step
        "step_roofline_ms": rl_ms, "step_roofline_bound": bound,
        "frac_of_step_roofline": rl_ms / ms_rank,
    })
    del dev, out
    # end to end through the host-buffer entry point (pinned buffers; the
    # copies both ways are inside the timed region)
    hp = {k: (torch.from_numpy(v).pin_memory() if v is not None else None) for k, v in inp.items()}
    hout = torch.empty(plan.out_shape, dtype=torch.float32).pin_memory()
    for _ in range(2):
        plan.forward_host(hp["x"], hp["w"], hp["b"], hp["gamma"], hp["beta"], hout, stream)
    barrier(world)
    e2e_times = []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        plan.forward_host(hp["x"], hp["w"], hp["b"], hp["gamma"], hp["beta"], hout, stream)
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(world, statistics.mean(e2e_times))
    assert plan.check_device(stream) == B.CN_OK
    h2d = sum(v.numel() * 4 for v in hp.values() if v is not None)
    e2e = {"value": world * flops / e2e_s / 1e9, "unit": "GFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * 4,
           "ms_per_step": e2e_s * 1e3, "steps": e2e_steps,
           "api": "conv_norm_forward_host (C ABI, pinned host buffers)"}
    plan.close()
    del hp, hout
    res = {"workload": spec["name"], "ms": ms, "ms_rank": ms_rank, "steps": steps,
           "gflops": job_rate(world, flops, ms) / 1e9, "flops_per_step": flops,
           "roofline_ms": rl_ms, "bound": bound, "frac": rl_ms / ms,
           "roofline": roofline, "e2e": e2e, "launches": nl, "kernels": info["kernel_names"],
           "contraction": contraction(info["kernel_names"]), "config": config_of(spec)}
    if clocks:
        res["clocks"] = clocks
    if cpu_target_s:
        rate, n, dt, thr = oracle_rate(spec, inp, target_s=cpu_target_s)
        res["cpu_baseline"] = {"value": rate, "unit": "GFLOP/s", "cores": thr, "kind": "oracle",
                               "sample": f"{n} of {spec['N']} samples, {dt:.1f} s"}
    return res


BACKWARD_METRIC = "fused conv+norm backward ms & GFLOP/s (dx and dw work), % of roofline (FP32 peak vs HBM)"
BACKWARD_WORKLOADS = ("conv2d_in_half_n32", "convt2d_g8_gelu_gn8_n32")


def backward_flops(s):
    """The gradients' own work: dx and dw are each one conv's multiply-adds
    (2 x the forward conv's FLOPs together); the conv output the backward
    recomputes is not counted."""
    return 2.0 * algorithmic_flops(s)


def backward_bytes(s):
    """Compulsory bytes of one backward: read x, w, dout (and b, gamma,
    beta), write dx, dw (and db, dgamma, dbeta)."""
    shp = wl.input_shapes(s)
    n = sum(math.prod(v) for v in shp.values() if v)
    return 4.0 * (2 * n + math.prod(out_shape(s)))


def measure_backward(B, torch, spec, pk, stream, flush, steps, warmup):
    """Backward step time (mean of `steps`, L2 flushed before each, CUDA
    events on the stream) through conv_norm_backward, for a full-output 2-D
    workload; dout is seeded N(0, 1)."""
    import numpy as np
    inp = wl.make_inputs(spec)
    dev = {k: (torch.from_numpy(v).cuda() if v is not None else None) for k, v in inp.items()}
    dout = torch.from_numpy(np.random.default_rng(spec["seed"] + 100).standard_normal(
        out_shape(spec)).astype(np.float32)).cuda()
    aff = bool(spec["affine"]) and spec["norm"] != "none"
    g = {"dx": torch.empty_like(dev["x"]), "dw": torch.empty_like(dev["w"]),
         "db": torch.empty_like(dev["b"]) if spec["has_bias"] else None,
         "dgamma": torch.empty(spec["C_out"], device="cuda") if aff else None,
         "dbeta": torch.empty(spec["C_out"], device="cuda") if aff else None}
    plan = B.BwdPlan(spec)

    def bwd():
        plan.backward(dev["x"], dev["w"], dev["b"], dev["gamma"] if aff else None,
                      dev["beta"] if aff else None, dout, g["dx"], g["dw"], g["db"], g["dgamma"],
                      g["dbeta"], stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            bwd()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    stream.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(min(2e9, 2e6 * steps + 2e7)))
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            bwd()
            e1.record(stream)
    stream.synchronize()
    assert plan.check_device(stream) == B.CN_OK
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    ws = plan.workspace_bytes()
    plan.close()
    flops, nbytes = backward_flops(spec), backward_bytes(spec)
    rl_ms = max(flops / (pk["fp32_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9)) * 1e3
    return {"workload": spec["name"], "ms": ms, "steps": steps, "gflops": flops / ms / 1e6,
            "flops_per_step": flops, "roofline_ms": rl_ms, "frac": rl_ms / ms,
            "bound": "alu" if flops / (pk["fp32_tflops"] * 1e12) >= nbytes / (pk["hbm_gbs"] * 1e9) else "hbm",
            "workspace_bytes": ws,
            "api": "conv_norm_backward (C ABI): conv recompute, plane sums, group coefficients, dA, "
                   "adjoint conv (dx), split-K correlation (dw), channel sums"}


def run_cuda(args, spec):
    import torch
    world, rank, local = dist_setup(args.gpus)
    from convolution_normalization_gb300 import build as cn_build
    if rank == 0:
        cn_build.build()
    barrier(world)
    from convolution_normalization_gb300 import binding as B

    torch.cuda.set_device(local)
    pk = peaks(torch.cuda.get_device_properties(local).multi_processor_count)
    stream = torch.cuda.Stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    if args.backward:
        r = measure_backward(B, torch, spec, pk, stream, flush, args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"metric": BACKWARD_METRIC, "value": r["gflops"], "unit": "GFLOP/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": "f32", "data": DATA, "config": config_of(spec),
                              "backward": r}), flush=True)
        return
    head = measure(B, torch, spec, pk, stream, flush, args.steps, args.warmup, world,
                   e2e_steps=max(3, min(args.steps, 30)),
                   cpu_target_s=None if (rank != 0 or args.no_cpu_baseline) else 12.0,
                   sampler=ClockSampler(torch.cuda.current_device()))

    line = {
        "metric": METRIC, "value": head["gflops"], "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": DATA, "config": head["config"], "contraction": head["contraction"],
        "roofline": head["roofline"],
        "gpu_launches": args.steps * head["launches"],
        "kernels": head["kernels"],
        "clocks": head["clocks"],
        "e2e": head["e2e"],
        "peaks": {k: pk[k] for k in ("hbm_gbs", "fp32_tflops", "bf16_tflops", "sm_max_mhz",
                                      "sms", "source")},
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if rank == 0 and not args.no_extras:
        extras = []
        for s2 in wl.WORKLOADS:
            if s2["name"] == spec["name"]:
                continue
            r = measure(B, torch, s2, pk, stream, flush, 30, 5, 1, e2e_steps=10,
                        cpu_target_s=None if args.no_cpu_baseline else 3.0)
            r.pop("config")
            extras.append(r)
        line["workloads"] = extras
        line["backward"] = [measure_backward(B, torch, wl.WORKLOAD_BY_NAME[n], pk, stream, flush, 20, 3)
                            for n in BACKWARD_WORKLOADS]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass of the workload instead (full-output 2-D workloads)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small cases for profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    spec = wl.WORKLOAD_BY_NAME[args.workload]
    if args.batch is not None:
        spec = wl.with_overrides(spec, N=args.batch, name=f"{spec['name']}_batch{args.batch}")
    if args.impl == "reference":
        run_reference(args, spec)
    else:
        run_cuda(args, spec)


if __name__ == "__main__":
    main()
