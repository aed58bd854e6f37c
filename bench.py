#!/usr/bin/env python
"""Benchmark of the MoE layer hot path on GB300: prints ONE JSON line.

A step is one pass of the whole path over one batch of synthetic input: router
(GEMM + score + top-k + gates), permute (histogram, scan, scatter), grouped
SwiGLU experts, combine, and for training workloads the full backward (combine
backward, SwiGLU backward, data and weight gradients of every GEMM, permute
backward, router backward with the auxiliary-loss gradient).

The default workload is the Qwen3-235B-shaped layer (T=16384 tokens, H=4096,
E=128 experts, top-8, F=1536) as a training step, balanced routing. Its
inputs (x 134 MB, expert weights 4.8 GB) are larger than the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (N>1, one process per GPU under torch.distributed.run): the path
does not shard across GPUs here; every rank runs an independent replica of the
layer (weak scaling, no collective on the data path); time is the max over
ranks and the value is the work of all ranks over that time.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer TFLOPS (fwd, fwd+bwd) & tokens/s on 1 GB300; % of BF16/HBM roofline"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_train")
    ap.add_argument("--seed", type=int, default=1234)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA Graph replay timing")
    ap.add_argument("--no-lib-peaks", action="store_true",
                    help="skip the vendor library's FP8/NVFP4 GEMM rates (low-precision fractions then take the "
                         "nominal ratios to the measured bf16 peak)")
    ap.add_argument("--force-balanced", action="store_true", help="force-balanced routing (cyclic assignment)")
    ap.add_argument("--no-mxfp8", action="store_true", help="skip the MXFP8 forward timing")
    ap.add_argument("--no-nvfp4", action="store_true", help="skip the NVFP4 grouped GEMM timing")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements (Mixtral, Qwen3, skewed Qwen3, DeepSeek-V3 shapes)")
    ap.add_argument("--recompute", action="store_true",
                    help="memory-saving training step (a and y_perm not kept; recomputed in the backward)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# algorithmic FLOPs and bytes
# ----------------------------------------------------------------------------
def layer_flops(ls, training):
    """Active FLOPs: router 2THE, routed experts 6HF per (token, expert) pair,
    shared expert 6HFs per token; the backward is twice the forward."""
    T, H, E, k, F = ls.T, ls.H, ls.E, ls.k, ls.F
    fwd = 2 * T * H * E + 6 * H * F * T * k + 6 * H * ls.F_shared * T
    return 3 * fwd if training else fwd


def stage_model(ls, training):
    """Per stage: (algorithmic FLOPs, algorithmic bytes) of one launch."""
    T, H, E, k, F = ls.T, ls.H, ls.E, ls.k, ls.F
    R = T * k
    Ep = ((E + 63) // 64) * 64
    yb = 2  # bf16 storage of y_perm (fp32 when inter_fp32)
    if ls.inter_fp32:
        yb = 4
    m = {
        "router": (2 * T * H * E, 2 * T * H + 2 * E * H + 8 * T * k + (4 * T * E if training else 0)),
        "permute": (0, 4 * T * k * 2 + 2 * T * H + 2 * R * H + 4 * T * k),
        "ffn1_gate_up": (2 * R * H * 2 * F, 2 * R * H + 2 * 2 * E * H * F + 2 * R * F + (4 * R * F if training else 0)),
        "ffn2_down": (2 * R * F * H, 2 * R * F + 2 * E * F * H + yb * R * H),
        "combine": (0, yb * R * H + 2 * T * H + 8 * T * k),
    }
    if ls.F_shared:
        Fs = ls.F_shared
        m["shared_gate_up"] = (2 * T * H * 2 * Fs, 2 * T * H + 4 * H * Fs + 2 * T * Fs)
        m["shared_down"] = (2 * T * Fs * H, 2 * T * Fs + 2 * Fs * H + yb * T * H)
    if training:
        rec = bool(ls.extra.get("recompute", False))  # memory-saving backward: no y_perm read, a re-written
        m.update({
            "combine_bwd": (0, 2 * T * H + (0 if rec else yb * R * H) + 2 * R * H + 8 * T * k),
            "router_bwd_elem": (0, 4 * T * E + 12 * T * k + 2 * T * 2 * Ep),
            "dgrad_down_swiglu": (2 * R * H * F, 2 * R * H + 2 * E * F * H + 4 * R * F + 4 * R * F
                                  + (2 * R * F if rec else 0)),
            "wgrad_down": (2 * R * F * H, 2 * R * F + 2 * R * H + 4 * E * F * H),
            "dgrad_gate_up": (2 * R * 2 * F * H, 4 * R * F + 4 * E * H * F + 2 * R * H),
            "wgrad_gate_up": (2 * R * H * 2 * F, 2 * R * H + 4 * R * F + 8 * E * H * F),
            "router_dgrad": (2 * T * 2 * Ep * H, 2 * T * 2 * Ep + 2 * E * H + 4 * T * H),
            "permute_bwd": (0, 2 * R * H + 4 * T * H + 2 * T * H + 4 * T * k),
            "router_wgrad": (2 * T * 2 * Ep * H, 2 * T * 2 * Ep + 2 * T * H + 4 * E * H),
            "aux_loss": (0, 4 * E * (T // 32 + 2)),
        })
    return m


TENSOR_STAGES = {"router", "ffn1_gate_up", "ffn2_down", "shared_gate_up", "shared_down", "dgrad_down_swiglu",
                 "wgrad_down", "dgrad_gate_up", "wgrad_gate_up", "router_dgrad", "router_wgrad"}


def kernel_table(stages, model, peaks):
    """Per stage: average ms per launch, launches, share of the stage time and
    the fraction of its roofline. A contraction whose arithmetic intensity
    (FLOP per algorithmic byte) is below the ridge point of the two measured
    peaks is bounded by HBM. Returns (table, {stage: [total ms, launches]})."""
    ridge = peaks["bf16_tflops_sustained"] * 1e3 / peaks["hbm_gbs"]  # FLOP per byte
    agg = {}
    for name, t in stages:
        a = agg.setdefault(name, [0.0, 0])
        a[0] += t
        a[1] += 1
    kernels = {}
    for name, (tot, n) in agg.items():
        avg = tot / n
        fl, by = model.get(name, (0, 0))
        ent = {"ms": round(avg, 4), "launches": n, "share": None}
        if name in TENSOR_STAGES and fl and (not by or fl / by >= ridge):
            ach = fl / (avg * 1e-3) / 1e12
            ent.update(bound="tensor", achieved_tflops=round(ach, 1),
                       frac=round(ach / peaks["bf16_tflops_sustained"], 4))
        elif by:
            ach = by / (avg * 1e-3) / 1e9
            ent.update(bound="hbm", achieved_gbs=round(ach, 1), frac=round(ach / peaks["hbm_gbs"], 4))
            if fl:
                ent["achieved_tflops"] = round(fl / (avg * 1e-3) / 1e12, 1)
        kernels[name] = ent
    total_stage = sum(v[0] for v in agg.values())
    for name in kernels:
        kernels[name]["share"] = round(agg[name][0] / total_stage, 4) if total_stage else None
    return kernels, agg


_READ_CEILING = {}


def device_ms(fn, reps=3):
    """Average device time of `fn()` over `reps` calls: CUDA events on the
    current stream, after one untimed call."""
    import torch

    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def library_gemm_rate(mm, n, reps_seconds, what):
    """Best of 10 launches (burst) and back to back for `reps_seconds`
    (sustained) of the library GEMM `mm()` of size n^3, as TFLOP/s; None where
    the call is unavailable."""
    import torch

    try:
        mm()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(10):
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        reps = max(10, int(reps_seconds * 1e3 / best))
        e0.record()
        for _ in range(reps):
            mm()
        e1.record()
        torch.cuda.synchronize()
        sus = e0.elapsed_time(e1) / reps
        fl = 2.0 * n ** 3
        return {"burst_tflops": round(fl / (best * 1e-3) / 1e12, 1),
                "sustained_tflops": round(fl / (sus * 1e-3) / 1e12, 1),
                "how": f"{what} {n}^3, best of 10 and {reps} back to back"}
    except Exception as ex:  # the library GEMM is missing on this build
        print(f"{what}: not measured: {ex}", file=sys.stderr)
        return None


def measured_fp8_peak(dev, seconds=2.0):
    """Rate of a dense FP8 GEMM from the vendor library (torch._scaled_mm:
    e4m3 x e4m3, per-tensor scales, bf16 out), measured the way the bf16 peaks
    beside it were."""
    import torch

    n = 8192
    g = torch.Generator(device=dev).manual_seed(11)
    a = (0.5 * torch.randn((n, n), generator=g, device=dev)).to(torch.float8_e4m3fn)
    b = (0.5 * torch.randn((n, n), generator=g, device=dev)).to(torch.float8_e4m3fn)
    one = torch.ones((), dtype=torch.float32, device=dev)
    return library_gemm_rate(lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16),
                             n, seconds, "torch._scaled_mm e4m3")


def measured_fp4_peak(dev, seconds=2.0):
    """Rate of a dense NVFP4 GEMM from the vendor library (torch._scaled_mm:
    e2m1 x e2m1 with an e4m3 scale per 16 elements, bf16 out); None where the
    library or this torch build does not offer it."""
    import torch

    if not hasattr(torch, "float4_e2m1fn_x2"):
        return None
    n = 8192
    g = torch.Generator(device=dev).manual_seed(12)
    a = torch.randint(0, 256, (n, n // 2), generator=g, dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
    b = torch.randint(0, 256, (n, n // 2), generator=g, dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
    sa = torch.ones(n * (n // 16), device=dev).to(torch.float8_e4m3fn)
    sb = torch.ones(n * (n // 16), device=dev).to(torch.float8_e4m3fn)
    return library_gemm_rate(lambda: torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16),
                             n, seconds, "torch._scaled_mm nvfp4")


def read_ceiling_gbs(nbytes, dev, reps=7):
    """Median rate of one moe_read_ceiling launch over `nbytes` (cold L2: a
    buffer larger than L2 is written before each launch): the rate at which a
    single kernel that reads that many bytes can stream them, launch ramp-up and
    tail included. The router reads x once; its fraction of this ceiling says
    how close it comes to a plain read of the same size."""
    import torch

    from route_permute_grouped_gb300 import ops

    nbytes = int(nbytes) // 16 * 16
    if nbytes in _READ_CEILING:
        return _READ_CEILING[nbytes]
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    sink = torch.zeros(4096, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ts = []
    for i in range(reps + 1):
        flush.fill_(i & 0xff)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ops.read_ceiling(buf, sink)
        b.record()
        torch.cuda.synchronize()
        if i:
            ts.append(a.elapsed_time(b))
    ts.sort()
    gbs = nbytes / (ts[len(ts) // 2] * 1e-3) / 1e9
    del buf, flush, sink
    _READ_CEILING[nbytes] = round(gbs, 1)
    return _READ_CEILING[nbytes]


_WRITE_CEILING = {}


def write_ceiling_gbs(dev, nbytes=1 << 30, reps=5):
    """Median rate of one moe_write_ceiling launch filling `nbytes` (8x the
    L2): the rate at which HBM absorbs a stream of writes, below the copy
    peak's read + write figure."""
    import torch

    from route_permute_grouped_gb300 import ops

    if nbytes in _WRITE_CEILING:
        return _WRITE_CEILING[nbytes]
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ts = []
    for i in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ops.write_ceiling(buf, i)
        b.record()
        torch.cuda.synchronize()
        if i:
            ts.append(a.elapsed_time(b))
    ts.sort()
    del buf
    _WRITE_CEILING[nbytes] = round(nbytes / (ts[len(ts) // 2] * 1e-3) / 1e9, 1)
    return _WRITE_CEILING[nbytes]


def add_read_ceiling(kernels, model, dev, ls=None):
    """The router's row gains the single-launch read ceiling of its bytes;
    the weight gradients' rows the rate of their fp32 output against the
    measured write ceiling (their output is 6.4 + 3.2 GB per Qwen3 step)."""
    if "router" in kernels and kernels["router"].get("achieved_gbs"):
        rc = read_ceiling_gbs(model["router"][1], dev)
        kernels["router"]["read_ceiling_gbs"] = rc
        kernels["router"]["frac_of_read_ceiling"] = round(kernels["router"]["achieved_gbs"] / rc, 4)
    if ls is not None and any(n in kernels for n in ("wgrad_gate_up", "wgrad_down")):
        wc = write_ceiling_gbs(dev)
        out = {"wgrad_gate_up": 8 * ls.E * ls.H * ls.F, "wgrad_down": 4 * ls.E * ls.F * ls.H}
        for name, nb in out.items():
            if name in kernels:
                gbs = nb / (kernels[name]["ms"] * 1e-3) / 1e9
                kernels[name].update(output_gbs=round(gbs, 1), write_ceiling_gbs=wc,
                                     frac_of_write_ceiling=round(gbs / wc, 4))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class Clocks:
    """nvidia-smi samples (every 50 ms) of the SM clock, its maximum, the power
    draw and the throttle reasons; only samples stamped inside the timed region
    (between mark_begin and mark_end) are kept."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # the sampler is running before the timed region starts
        except Exception:
            self.proc = None

    def mark_begin(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows, every = [], []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            every.append(parts)
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            if self.t0 is not None and self.t1 is not None and not (self.t0 <= ts <= self.t1):
                continue
            rows.append(parts)
        os.unlink(self.path)
        rows = rows or every  # unparsable stamps: keep every sample
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[6 + j].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(ls, d, seed, n_experts=4, n_router_tokens=1024, max_rows=None):
    """Prepare a bounded sample of the same workload for the fp64 oracle: the
    rows of `n_experts` seeded experts (at most `max_rows` each; forward +
    backward of those experts) and the router over `n_router_tokens` tokens.
    Returns (fn, flops, description): fn() runs the sample once."""
    import numpy as np
    import torch

    import oracle as O

    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    x = f64(d["x"])
    w_r = f64(d["router_w"])
    lb = None if d["logit_bias"] is None else f64(d["logit_bias"])
    rt = O.route(x, w_r, ls.k, ls.score, None if d["expert_bias"] is None else f64(d["expert_bias"]), lb,
                 ls.n_groups, ls.topk_groups, ls.gate_scale, force_balanced=ls.force_balanced)
    rng = np.random.default_rng(seed)
    experts = sorted(rng.choice(ls.E, size=min(n_experts, ls.E), replace=False).tolist())
    data = []
    rows_total = 0
    for e in experts:
        tt, ii = np.nonzero(rt["topk_idx"] == e)
        if max_rows is not None:
            tt, ii = tt[:max_rows], ii[:max_rows]
        W = (f64(d["W1"][e]), f64(d["W3"][e]), f64(d["W2"][e]))
        xr = x[tt]
        dO = f64(d["dO"][torch.from_numpy(tt).to(d["dO"].device)]) if d["dO"] is not None else None
        data.append((xr, W, rt["topk_gate"][tt, ii], dO))
        rows_total += len(tt)
    xs = x[:n_router_tokens]
    training = ls.aux_coeff > 0 or d["dO"] is not None

    eb = None if d["expert_bias"] is None else f64(d["expert_bias"])

    def fn():
        O.route(xs, w_r, ls.k, ls.score, eb, lb, ls.n_groups, ls.topk_groups, ls.gate_scale,
                force_balanced=ls.force_balanced)
        for xr, W, g, dO in data:
            h1, h3, a, out = O.swiglu_expert(xr, *W)
            if training and dO is not None:
                dyr = O.bf16_rne(g[:, None] * dO)
                O.expert_backward(xr, O.bf16_rne(h1), O.bf16_rne(h3), a, dyr, *W)

    mult = 3 if training else 1
    flops = mult * (2 * len(xs) * ls.H * ls.E + 6 * ls.H * ls.F * rows_total)
    desc = (f"fp64 numpy oracle: router over {len(xs)} tokens + {'fwd+bwd' if training else 'fwd'} of "
            f"{len(experts)} seeded experts ({rows_total} routed rows) of the {ls.name} layer")
    return fn, flops, desc


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def time_oracle(fn, flops, reps):
    t0 = time.perf_counter()
    for _ in range(reps):
        fn()
    dt = (time.perf_counter() - t0) / reps
    return flops / dt / 1e12, dt


# ----------------------------------------------------------------------------
def max_over_ranks(x, world, device):
    """The maximum of a per-rank value over all ranks (a step time: the job
    is as fast as its slowest replica). Identity on one process."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step, ms_per_step, world):
    """Whole-job TFLOPS: the work of every rank over the max-over-ranks step
    time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def run_reference(args, ls):
    import torch

    from route_permute_grouped_gb300 import synth

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = synth.make_layer(ls, seed=args.seed, device=dev, training=ls.aux_coeff > 0)
    fn, flops, desc = oracle_sample(ls, d, args.seed)
    for _ in range(args.warmup):
        fn()
    tflops, dt = time_oracle(fn, flops, args.steps)
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tflops, 6), "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(ls),
        "cpu_baseline": {"value": round(tflops, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(tflops, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(ls):
    return {"workload": f"{ls.name}: MoE layer T={ls.T} H={ls.H} E={ls.E} k={ls.k} F={ls.F}"
                        + (f" Fs={ls.F_shared}" if ls.F_shared else "")
                        + f" {ls.score} top-{ls.k}" + (f" groups {ls.n_groups}/{ls.topk_groups}" if ls.n_groups > 1 else "")
                        + (" force-balanced" if ls.force_balanced else (f" zipf {ls.skew}" if ls.skew else " balanced"))
                        + (" fwd+bwd" if ls.aux_coeff > 0 else " fwd"),
            "tokens": ls.T, "hidden": ls.H, "experts": ls.E, "top_k": ls.k, "ffn": ls.F,
            "memory_saving": bool(ls.extra.get("recompute", False)),
            "l2": (f"inputs larger than the 129 MB L2 (x {2 * ls.T * ls.H / 1e6:.0f} MB, expert weights "
                   f"{6 * ls.E * ls.H * ls.F / 1e9:.2f} GB); no flush")}


def run_ours(args, ls, rank, world, local_rank):
    import numpy as np
    import torch

    from route_permute_grouped_gb300 import build, ops, synth

    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    training = ls.aux_coeff > 0
    d = synth.make_layer(ls, seed=args.seed + rank, device=dev, training=training)
    cfg = ops.config_from_shape(ls)
    ws = ops.workspace(cfg, training, dev)
    saved = ops.alloc_saved(cfg, dev, recompute=args.recompute) if training else None
    grads = ops.alloc_grads(cfg, dev) if training else None
    y = torch.empty((ls.T, ls.H), dtype=torch.bfloat16, device=dev)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None

    def fwd():
        ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                      saved=saved, ws=ws, y=y)

    def step():
        fwd()
        if training:
            ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws, grads=grads)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = ops.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---------------- timed region: K whole steps
    cap = args.steps * 32 + 64
    clocks = Clocks(local_rank)
    barrier()
    clocks.start()
    clocks.mark_begin()
    l0 = ops.launch_count()
    ops.profile_start(cap)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    ops.profile_stop()
    barrier()
    clk = clocks.stop()
    launches = ops.launch_count() - l0
    ms = e0.elapsed_time(e1) / args.steps
    stages = ops.profile_read(cap)
    ms = max_over_ranks(ms, world, dev)
    assert ops.device_status(ws) == 0

    # ---------------- forward-only timing (same inputs)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    for _ in range(args.steps):
        fwd()
    f1.record()
    torch.cuda.synchronize()
    ms_fwd = f0.elapsed_time(f1) / args.steps
    ms_fwd = max_over_ranks(ms_fwd, world, dev)

    # ---------------- end to end through the C ABI with host buffers (right after
    # the device-timed steps, so that both see the GPU in the same state)
    flops_step = layer_flops(ls, training)
    e2e = None
    if not args.no_e2e:
        hx = d["x"].cpu().pin_memory()
        hdO = d["dO"].cpu().pin_memory() if training else None
        hy = torch.empty((ls.T, ls.H), dtype=torch.bfloat16).pin_memory()
        hdx = torch.empty((ls.T, ls.H), dtype=torch.bfloat16).pin_memory() if training else None
        haux = torch.empty(1, dtype=torch.float32).pin_memory()
        # every step copies its inputs in from pinned host memory and its
        # results out; the copies run on two copy streams, double-buffered on
        # the device, so they overlap the neighbouring steps' compute. In a
        # training step they run beside the backward's GEMMs (compute-bound):
        # once step i's forward is done, step i-1's results go out and step
        # i+1's inputs come in, away from the forward's memory-bound kernels
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        xd = [torch.empty_like(d["x"]) for _ in range(2)]
        dOd = [torch.empty_like(d["dO"]) for _ in range(2)] if training else None
        ys = [y, torch.empty_like(y)]
        gbuf = None
        if training:
            gbuf = [grads, dict(grads, dx=torch.empty_like(grads["dx"]), aux_loss=torch.zeros_like(grads["aux_loss"]))]
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b on the device
        ev_used = [torch.cuda.Event() for _ in range(2)]  # compute finished with inputs / outputs of b
        ev_read = [torch.cuda.Event() for _ in range(2)]  # outputs of b copied to the host
        ev_fwd = torch.cuda.Event()                       # the current step's forward is done

        def issue_h2d(i, after=None):
            b = i % 2
            if after is not None:
                s_in.wait_event(after)
            with torch.cuda.stream(s_in):
                xd[b].copy_(hx, non_blocking=True)
                if training:
                    dOd[b].copy_(hdO, non_blocking=True)
                ev_in[b].record(s_in)

        def issue_d2h(i, after):
            b = i % 2
            s_out.wait_event(after)
            with torch.cuda.stream(s_out):
                hy.copy_(ys[b], non_blocking=True)
                if training:
                    hdx.copy_(gbuf[b]["dx"], non_blocking=True)
                    haux.copy_(gbuf[b]["aux_loss"], non_blocking=True)
                ev_read[b].record(s_out)

        def e2e_step(i, n):
            b = i % 2
            comp.wait_event(ev_in[b])
            if i >= 2:
                comp.wait_event(ev_read[b])
            ops.layer_fwd(cfg, xd[b], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                          Ws, saved=saved, ws=ws, y=ys[b])
            if training:
                ev_fwd.record(comp)  # step i-1 is complete as well
                if i >= 1:
                    issue_d2h(i - 1, ev_fwd)
                if i + 1 < n:
                    issue_h2d(i + 1, ev_fwd)
                ops.layer_bwd(cfg, dOd[b], xd[b], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws,
                              grads=gbuf[b])
            ev_used[b].record(comp)
            if not training:
                issue_d2h(i, ev_used[b])
                if i + 2 < n:
                    issue_h2d(i + 2, ev_used[b])

        def e2e_run(n):
            issue_h2d(0)
            if n > 1 and not training:
                issue_h2d(1)
            for i in range(n):
                e2e_step(i, n)
            if training:
                issue_d2h(n - 1, ev_used[(n - 1) % 2])
            comp.wait_event(ev_read[(n - 1) % 2])  # the last results are on the host

        e2e_run(2)
        torch.cuda.synchronize()
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(comp)
        s_in.wait_stream(comp)  # the first copies start inside the timed region
        e2e_run(args.steps)
        g1.record(comp)
        torch.cuda.synchronize()
        ms_e2e = g0.elapsed_time(g1) / args.steps
        ms_e2e = max_over_ranks(ms_e2e, world, dev)
        h2d = hx.numel() * 2 + (hdO.numel() * 2 if training else 0)
        d2h = hy.numel() * 2 + ((hdx.numel() * 2 + 4) if training else 0)
        e2e = {"value": round(job_throughput(flops_step, ms_e2e, world), 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4)}

        # the host link alone, after the end-to-end run: one step's input
        # copies, its output copies, and both at once (an end-to-end step is no
        # shorter than the last, whatever the overlap)
        def link_ms(inputs, outputs, reps=3):
            torch.cuda.synchronize()
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(comp)
            s_in.wait_stream(comp)
            s_out.wait_stream(comp)
            for _ in range(reps):
                if inputs:
                    with torch.cuda.stream(s_in):
                        xd[0].copy_(hx, non_blocking=True)
                        if training:
                            dOd[0].copy_(hdO, non_blocking=True)
                if outputs:
                    with torch.cuda.stream(s_out):
                        hy.copy_(ys[0], non_blocking=True)
                        if training:
                            hdx.copy_(gbuf[0]["dx"], non_blocking=True)
            comp.wait_stream(s_in)
            comp.wait_stream(s_out)
            c1.record(comp)
            torch.cuda.synchronize()
            return c0.elapsed_time(c1) / reps

        ms_in, ms_out, ms_both = link_ms(True, False), link_ms(False, True), link_ms(True, True)
        e2e["host_link"] = {"h2d_gbs": round(h2d / (ms_in * 1e-3) / 1e9, 1),
                            "d2h_gbs": round(d2h / (ms_out * 1e-3) / 1e9, 1),
                            "copies_alone_ms": round(ms_both, 4)}

    # ---------------- the same step captured once as a CUDA graph and replayed
    # (device-side offsets: no host synchronisation inside a step)
    graph = None
    if not args.no_graph:
        gs = torch.cuda.Stream(device=dev)
        gs.wait_stream(torch.cuda.current_stream())
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            step()
        torch.cuda.current_stream().wait_stream(gs)
        for _ in range(2):
            cg.replay()
        barrier()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record()
        for _ in range(args.steps):
            cg.replay()
        q1.record()
        torch.cuda.synchronize()
        assert ops.device_status(ws) == 0
        ms_graph = max_over_ranks(q0.elapsed_time(q1) / args.steps, world, dev)
        graph = {"value": round(job_throughput(layer_flops(ls, training), ms_graph, world), 2), "unit": "TFLOPS",
                 "ms_per_step": round(ms_graph, 4)}

    # ---------------- the forward with MXFP8 expert GEMMs (same inputs; the
    # weights quantised once, outside the timed region, as a trained model's
    # would be)
    peaks = load_peaks()
    mx = None
    # FP8 dense peak: the vendor FP8 GEMM's sustained rate measured in this
    # run, else the measured sustained bf16 peak times the nominal fp8 : bf16
    # ratio of the tensor cores (2)
    fp8_meas = (measured_fp8_peak(dev) if not args.no_mxfp8 and not args.no_lib_peaks and ls.H % 128 == 0
                and ls.F % 128 == 0 else None)
    if fp8_meas is not None:
        peak8 = fp8_meas["sustained_tflops"]
        peak8_src = "measured in this run: " + fp8_meas["how"] + " (sustained)"
    else:
        peak8 = 2 * peaks["bf16_tflops_sustained"]
        peak8_src = f"{peaks['source']} bf16_tflops_sustained x 2 (nominal fp8:bf16 ratio)"
    if not args.no_mxfp8 and ls.H % 128 == 0 and ls.F % 128 == 0:
        mxw = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
        wsm = ops.mx_workspace(cfg, dev)
        ym = torch.empty_like(y)

        def fwd_mx():
            ops.layer_fwd_mxfp8(cfg, d["x"], d["router_w"], mxw, d["expert_bias"], d["logit_bias"], Ws=Ws, ws=wsm,
                                y=ym)

        for _ in range(max(3, args.warmup)):
            fwd_mx()
        barrier()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ops.profile_start(args.steps * 8 + 8)
        m0.record()
        for _ in range(args.steps):
            fwd_mx()
        m1.record()
        torch.cuda.synchronize()
        ops.profile_stop()
        assert ops.device_status(wsm) == 0
        ms_mx = max_over_ranks(m0.elapsed_time(m1) / args.steps, world, dev)
        mx_stages = {}
        for name, t in ops.profile_read(args.steps * 8 + 8):
            mx_stages.setdefault(name, []).append(t)
        R = ls.T * ls.k
        mk = {}
        for name, fl in (("ffn1_gate_up", 2 * R * ls.H * 2 * ls.F), ("ffn2_down", 2 * R * ls.F * ls.H)):
            if name in mx_stages:
                avg = sum(mx_stages[name]) / len(mx_stages[name])
                ach = fl / (avg * 1e-3) / 1e12
                mk[name] = {"ms": round(avg, 4), "bound": "tensor", "achieved_tflops": round(ach, 1),
                            "frac": round(ach / peak8, 4)}
        for name in ("router", "permute", "combine"):
            if name in mx_stages:
                mk[name] = {"ms": round(sum(mx_stages[name]) / len(mx_stages[name]), 4)}
        mx = {"value": round(job_throughput(layer_flops(ls, False), ms_mx, world), 2), "unit": "TFLOPS",
              "ms_per_step": round(ms_mx, 4), "dtype": "mxfp8 (e4m3, e8m0 scale per 32 along K)",
              "vs_bf16_fwd": round(ms_fwd / ms_mx, 3), "kernels": mk, "peak_fp8_tflops": round(peak8, 1),
              "peak_source": peak8_src, "fp8_gemm_measured": fp8_meas,
              "peak_fp8_nominal_ratio_tflops": round(2 * peaks["bf16_tflops_sustained"], 1)}
        del mxw, wsm, ym

    # ---------------- the MXFP8 training step: forward saving for the
    # backward, backward with MXFP8 data-gradient GEMMs (weights quantised
    # once, outside the timed region; the gradient buffers of the bf16 step
    # reused)
    mxt = None
    if training and not args.no_mxfp8 and ls.H % 128 == 0 and ls.F % 128 == 0 and not ls.F_shared:
        mxw = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
        mxbw = ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
        wst = ops.mx_train_workspace(cfg, dev)
        svm = ops.alloc_saved_mxfp8(cfg, dev)
        ym = torch.empty_like(y)

        def step_mx():
            ops.layer_fwd_mxfp8_train(cfg, d["x"], d["router_w"], mxw, svm, d["expert_bias"], d["logit_bias"],
                                      ws=wst, y=ym)
            ops.layer_bwd_mxfp8(cfg, d["dO"], d["x"], d["router_w"], mxbw, svm, ws=wst, grads=grads)

        for _ in range(max(3, args.warmup)):
            step_mx()
        barrier()
        cap_t = args.steps * 40 + 64
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ops.profile_start(cap_t)
        t0.record()
        for _ in range(args.steps):
            step_mx()
        t1.record()
        torch.cuda.synchronize()
        ops.profile_stop()
        assert ops.device_status(wst) == 0
        ms_mxt = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
        st_mx = {}
        for name, t in ops.profile_read(cap_t):
            st_mx.setdefault(name, []).append(t)
        R = ls.T * ls.k
        tk = {}
        for name, fl, pk in (("ffn1_gate_up", 2 * R * ls.H * 2 * ls.F, peak8), ("ffn2_down", 2 * R * ls.F * ls.H, peak8),
                             ("mx_dgrad_down_swiglu", 2 * R * ls.H * ls.F, peak8),
                             ("mx_dgrad_gate_up", 2 * R * 2 * ls.F * ls.H, peak8),
                             ("wgrad_down", 2 * R * ls.F * ls.H, peaks["bf16_tflops_sustained"]),
                             ("wgrad_gate_up", 2 * R * ls.H * 2 * ls.F, peaks["bf16_tflops_sustained"])):
            if name in st_mx:
                # per step (the gate/up weight gradient is two launches: dW1, dW3)
                avg = sum(st_mx[name]) / args.steps
                ach = fl / (avg * 1e-3) / 1e12
                tk[name] = {"ms": round(avg, 4), "bound": "tensor", "achieved_tflops": round(ach, 1),
                            "frac": round(ach / pk, 4)}
        for name in ("router", "permute", "combine", "combine_bwd", "router_bwd_elem", "permute_bwd"):
            if name in st_mx:
                tk[name] = {"ms": round(sum(st_mx[name]) / args.steps, 4)}
        # the same step with the weight gradients in MXFP8 too (operands
        # quantised along each expert's tokens)
        def step_mxw():
            ops.layer_fwd_mxfp8_train(cfg, d["x"], d["router_w"], mxw, svm, d["expert_bias"], d["logit_bias"],
                                      ws=wst, y=ym)
            ops.layer_bwd_mxfp8(cfg, d["dO"], d["x"], d["router_w"], mxbw, svm, ws=wst, grads=grads, mx_wgrad=True)

        for _ in range(max(3, args.warmup)):
            step_mxw()
        barrier()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ops.profile_start(cap_t)
        w0.record()
        for _ in range(args.steps):
            step_mxw()
        w1.record()
        torch.cuda.synchronize()
        ops.profile_stop()
        assert ops.device_status(wst) == 0
        ms_mxw = max_over_ranks(w0.elapsed_time(w1) / args.steps, world, dev)
        st_w = {}
        for name, t in ops.profile_read(cap_t):
            st_w.setdefault(name, []).append(t)
        wk = {}
        for name, fl in (("wgrad_down", 2 * R * ls.F * ls.H), ("wgrad_gate_up", 2 * R * ls.H * 2 * ls.F)):
            if name in st_w:
                avg = sum(st_w[name]) / args.steps
                ach = fl / (avg * 1e-3) / 1e12
                wk[name] = {"ms": round(avg, 4), "bound": "tensor", "achieved_tflops": round(ach, 1),
                            "frac": round(ach / peak8, 4)}
        if "mx_quantize_tokens" in st_w:
            # a, dy_perm, x_perm, dh1, dh3 read (bf16), their padded transposed codes written
            avg = sum(st_w["mx_quantize_tokens"]) / args.steps
            nbytes = 3 * R * (2 * ls.H + 3 * ls.F)
            gbs = nbytes / (avg * 1e-3) / 1e9
            wk["mx_quantize_tokens"] = {"ms": round(avg, 4), "bound": "hbm", "achieved_gbs": round(gbs, 1),
                                        "frac": round(gbs / peaks["hbm_gbs"], 4)}
        mxt_w = {"value": round(job_throughput(layer_flops(ls, True), ms_mxw, world), 2), "unit": "TFLOPS",
                 "ms_per_step": round(ms_mxw, 4), "vs_bf16_step": round(ms / ms_mxw, 3), "kernels": wk}
        # the weight copies (forward and data-gradient operands) that a
        # training loop refreshes once per optimizer step: not in ms_per_step
        wq_mx = max_over_ranks(device_ms(lambda: (ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"]),
                                                  ops.mx_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"]))),
                               world, dev)
        mxt = {"value": round(job_throughput(layer_flops(ls, True), ms_mxt, world), 2), "unit": "TFLOPS",
               "ms_per_step": round(ms_mxt, 4), "weight_quant_ms": round(wq_mx, 4),
               "ms_per_step_with_weight_quant": round(ms_mxt + wq_mx, 4),
               "dtype": "mxfp8 forward and data-gradient GEMMs, bf16 weight gradients (fp32 out)",
               "vs_bf16_step": round(ms / ms_mxt, 3), "kernels": tk, "peak_fp8_tflops": round(peak8, 1),
               "peak_source": peak8_src, "mxfp8_weight_gradients": mxt_w}
        del mxw, mxbw, wst, svm, ym

    # ---------------- the NVFP4 grouped expert GEMM on the down projection's
    # shape: rows grouped by expert as the forward grouped them (its offsets),
    # the layer's W2 (quantised beforehand), activations quantised per call
    nv = None
    if not args.no_nvfp4 and ls.F % 256 == 0 and ls.H % 8 == 0 and training:
        R = ls.T * ls.k
        nvw = ops.nv_quantize_weights(d["W2"])
        gen = torch.Generator(device=dev).manual_seed(args.seed + 7)
        a_in = torch.randn((R, ls.F), generator=gen, device=dev).to(torch.bfloat16)
        wsn = ops.nv_workspace(ls.E, R, ls.F, dev)
        yn = torch.empty((R, ls.H), dtype=torch.bfloat16, device=dev)
        offs = saved["offsets"]

        def gemm_nv():
            ops.nv_grouped_gemm(a_in, offs, nvw, ws=wsn, y=yn)

        for _ in range(max(3, args.warmup)):
            gemm_nv()
        barrier()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ops.profile_start(args.steps * 4 + 4)
        n0.record()
        for _ in range(args.steps):
            gemm_nv()
        n1.record()
        torch.cuda.synchronize()
        ops.profile_stop()
        assert ops.device_status(wsn) == 0
        ms_nv = max_over_ranks(n0.elapsed_time(n1) / args.steps, world, dev)
        st_nv = {}
        for name, t in ops.profile_read(args.steps * 4 + 4):
            st_nv.setdefault(name, []).append(t)
        fl = 2 * R * ls.F * ls.H
        # FP4 dense peak: the vendor NVFP4 GEMM's sustained rate measured in
        # this run, else the measured sustained bf16 peak times the nominal
        # fp4 : bf16 ratio (13.5 / 2.25)
        fp4_meas = None if args.no_lib_peaks else measured_fp4_peak(dev)
        if fp4_meas is not None:
            peak4 = fp4_meas["sustained_tflops"]
            peak4_src = "measured in this run: " + fp4_meas["how"] + " (sustained)"
        else:
            peak4 = 6 * peaks["bf16_tflops_sustained"]
            peak4_src = f"{peaks['source']} bf16_tflops_sustained x 6 (nominal fp4:bf16 ratio 13.5/2.25)"
        g_ms = sum(st_nv.get("nv_gemm", [0])) / max(1, len(st_nv.get("nv_gemm", [0])))
        q_ms = sum(st_nv.get("nv_quantize", [0])) / max(1, len(st_nv.get("nv_quantize", [0])))
        nv = {"shape": f"grouped {R} x {ls.F} x {ls.H} (down projection, {ls.E} experts)",
              "ms_per_call": round(ms_nv, 4), "value": round(fl / (ms_nv * 1e-3) / 1e12, 1), "unit": "TFLOPS",
              "gemm_ms": round(g_ms, 4), "quantize_ms": round(q_ms, 4),
              "gemm": {"bound": "tensor", "achieved_tflops": round(fl / (g_ms * 1e-3) / 1e12, 1) if g_ms else None,
                       "frac": round(fl / (g_ms * 1e-3) / 1e12 / peak4, 4) if g_ms else None},
              "dtype": "nvfp4 (e2m1, e4m3 scale per 16 along K, fp32 tensor scale)", "peak_fp4_tflops": round(peak4, 1),
              "peak_source": peak4_src, "fp4_gemm_measured": fp4_meas,
              "peak_fp4_nominal_ratio_tflops": round(6 * peaks["bf16_tflops_sustained"], 1)}
        del nvw, a_in, wsn, yn
        # the layer forward with NVFP4 expert GEMMs (same inputs)
        nlw = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
        yl = torch.empty_like(y)
        for _ in range(max(3, args.warmup)):
            ops.layer_fwd_nvfp4(cfg, d["x"], d["router_w"], nlw, d["expert_bias"], d["logit_bias"], y=yl)
        barrier()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record()
        for _ in range(args.steps):
            ops.layer_fwd_nvfp4(cfg, d["x"], d["router_w"], nlw, d["expert_bias"], d["logit_bias"], y=yl)
        l1.record()
        torch.cuda.synchronize()
        ms_nl = max_over_ranks(l0.elapsed_time(l1) / args.steps, world, dev)
        nv["layer_fwd"] = {"value": round(job_throughput(layer_flops(ls, False), ms_nl, world), 2), "unit": "TFLOPS",
                           "ms_per_step": round(ms_nl, 4), "vs_bf16_fwd": round(ms_fwd / ms_nl, 3)}
        del nlw, yl
        # the NVFP4 training step: forward saving for the backward, backward
        # with NVFP4 data-gradient GEMMs (weights quantised once, outside the
        # timed region; bf16 weight gradients into the bf16 step's buffers)
        if not ls.F_shared:
            nlw = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
            nbw = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
            wsn = ops.nv_train_workspace(cfg, dev)
            svn = ops.alloc_saved(cfg, dev)
            yl = torch.empty_like(y)

            def step_nv():
                ops.layer_fwd_nvfp4_train(cfg, d["x"], d["router_w"], nlw, svn, d["expert_bias"], d["logit_bias"],
                                          ws=wsn, y=yl)
                ops.layer_bwd_nvfp4(cfg, d["dO"], d["x"], d["router_w"], nbw, svn, ws=wsn, grads=grads)

            for _ in range(max(3, args.warmup)):
                step_nv()
            barrier()
            cap_n = args.steps * 48 + 64
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ops.profile_start(cap_n)
            s0.record()
            for _ in range(args.steps):
                step_nv()
            s1.record()
            torch.cuda.synchronize()
            ops.profile_stop()
            assert ops.device_status(wsn) == 0
            ms_nt = max_over_ranks(s0.elapsed_time(s1) / args.steps, world, dev)
            st_nt = {}
            for name, t in ops.profile_read(cap_n):
                st_nt.setdefault(name, []).append(t)
            nk = {}
            for name, fl, pk in (("ffn1_gate_up", 2 * R * ls.H * 2 * ls.F, peak4),
                                 ("ffn2_down", 2 * R * ls.F * ls.H, peak4),
                                 ("nv_dgrad_down", 2 * R * ls.H * ls.F, peak4),
                                 ("nv_dgrad_gate_up", 2 * R * 2 * ls.F * ls.H, peak4),
                                 ("wgrad_down", 2 * R * ls.F * ls.H, peaks["bf16_tflops_sustained"]),
                                 ("wgrad_gate_up", 2 * R * ls.H * 2 * ls.F, peaks["bf16_tflops_sustained"])):
                if name in st_nt:
                    avg = sum(st_nt[name]) / args.steps
                    ach = fl / (avg * 1e-3) / 1e12
                    nk[name] = {"ms": round(avg, 4), "bound": "tensor", "achieved_tflops": round(ach, 1),
                                "frac": round(ach / pk, 4)}
            if "nv_swiglu_bwd" in st_nt:
                # da fp32 and h13 read, dh13 written (bf16)
                avg = sum(st_nt["nv_swiglu_bwd"]) / args.steps
                gbs = 12 * R * ls.F / (avg * 1e-3) / 1e9
                nk["nv_swiglu_bwd"] = {"ms": round(avg, 4), "bound": "hbm", "achieved_gbs": round(gbs, 1),
                                       "frac": round(gbs / peaks["hbm_gbs"], 4)}
            for name in ("nv_quantize", "router", "permute", "combine", "combine_bwd", "router_bwd_elem",
                         "permute_bwd"):
                if name in st_nt:
                    nk[name] = {"ms": round(sum(st_nt[name]) / args.steps, 4)}
            # the weight copies a training loop refreshes once per optimizer
            # step (one call: the per-expert maxima once, then both copies'
            # codes): not in ms_per_step
            wq_nv = max_over_ranks(device_ms(lambda: ops.nv_quantize_train_weights(cfg, d["W1"], d["W3"], d["W2"])),
                                   world, dev)
            nv["train_step"] = {"value": round(job_throughput(layer_flops(ls, True), ms_nt, world), 2),
                                "unit": "TFLOPS", "ms_per_step": round(ms_nt, 4), "vs_bf16_step": round(ms / ms_nt, 3),
                                "weight_quant_ms": round(wq_nv, 4),
                                "ms_per_step_with_weight_quant": round(ms_nt + wq_nv, 4),
                                "dtype": "nvfp4 forward and data-gradient GEMMs, bf16 weight gradients (fp32 out)",
                                "kernels": nk}
            del nlw, nbw, wsn, svn, yl

    # ---------------- per-stage table and roofline of the dominant kernel
    model = stage_model(ls, training)
    kernels, agg = kernel_table(stages, model, peaks)
    add_read_ceiling(kernels, model, dev, ls)
    dom = max(agg, key=lambda n: agg[n][0])
    dk = kernels[dom]
    fl, by = model[dom]
    if dk.get("bound") == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": dk["achieved_tflops"],
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s", "frac": dk["frac"],
                "traffic": None, "algorithmic_flops_per_launch": fl, "avg_launch_ms": dk["ms"],
                "peak_source": f"{peaks['source']} bf16_tflops_sustained (kernel timed inside a long step)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": dk["achieved_gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": dk["frac"], "traffic": None, "algorithmic_bytes_per_launch": by,
                "avg_launch_ms": dk["ms"], "peak_source": f"{peaks['source']} hbm_gbs"}
    traffic = load_traffic(dom)
    if traffic is not None:
        roof["traffic"] = traffic

    flops_step = layer_flops(ls, training)
    value = job_throughput(flops_step, ms, world)
    fwd_value = job_throughput(layer_flops(ls, False), ms_fwd, world)

    # ---------------- CPU baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fn, fl_s, desc = oracle_sample(ls, d, args.seed)
        reps = 1
        t0 = time.perf_counter()
        fn()
        one = time.perf_counter() - t0
        reps = max(1, min(10, int(15.0 / max(one, 1e-3))))
        tflops, dt = time_oracle(fn, fl_s, reps)
        cpu = {"value": round(tflops, 6), "unit": "TFLOPS", "cores": blas_threads(), "kind": "oracle",
               "sample": desc + f"; {reps} repetitions, {dt:.2f} s each"}

    # ---------------- every layer configuration, each as its own measurement
    configs = None
    if not args.no_configs:
        configs = {}
        for name in CONFIG_LINES:
            configs[name] = measure_config(name, args, rank, world, dev, peaks)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(ls),
            "tokens_per_s": round(world * ls.T / (ms * 1e-3), 1),
            "fwd": {"value": round(fwd_value, 2), "unit": "TFLOPS", "ms_per_step": round(ms_fwd, 4),
                    "tokens_per_s": round(world * ls.T / (ms_fwd * 1e-3), 1)},
            "graph": graph, "mxfp8_fwd": mx, "mxfp8_train": mxt, "nvfp4_grouped_gemm": nv, "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk, "configs": configs,
        }
        print(json.dumps(line), flush=True)


# The layer configurations each measured as a sub-object of the one bench line
# (their shapes are route_permute_grouped_gb300.synth's): the Mixtral-8x7B-,
# Qwen3-235B- (balanced and Zipf-skewed) and DeepSeek-V3-shaped forwards and
# the skewed Qwen3 training step.
CONFIG_LINES = ("mixtral", "qwen3", "qwen3_skew", "qwen3_skew_train", "dsv3")


def measure_config(name, args, rank, world, dev, peaks):
    """One layer configuration: the step (forward, or forward + backward for a
    training workload) timed with CUDA events over inputs larger than L2,
    per-stage roofline fractions, the expert-count histogram summary, and the
    fp64 oracle on a bounded sample of the same workload (rank 0, N = 1)."""
    import numpy as np
    import torch

    from route_permute_grouped_gb300 import ops, synth

    ls = synth.shape(name)
    training = ls.aux_coeff > 0
    d = synth.make_layer(ls, seed=args.seed + rank, device=dev, training=training)
    cfg = ops.config_from_shape(ls)
    ws = ops.workspace(cfg, training, dev)
    saved = ops.alloc_saved(cfg, dev) if training else None
    grads = ops.alloc_grads(cfg, dev) if training else None
    y = torch.empty((ls.T, ls.H), dtype=torch.float32 if cfg.out_fp32 else torch.bfloat16, device=dev)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None

    def step():
        ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                      saved=saved, ws=ws, y=y)
        if training:
            ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws,
                          grads=grads, Ws=Ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if ops.device_status(ws) != 0:
        raise RuntimeError(f"{name}: device status after warm-up")
    steps = max(3, min(args.steps, 10))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    cap = steps * 40 + 64
    ops.profile_start(cap)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ops.profile_stop()
    assert ops.device_status(ws) == 0
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)
    kernels, agg = kernel_table(ops.profile_read(cap), stage_model(ls, training), peaks)
    add_read_ceiling(kernels, stage_model(ls, training), dev, ls)
    # the expert-count histogram of this routing (one training-style forward
    # keeps the counts)
    sv = saved if saved is not None else ops.alloc_saved(cfg, dev)
    wsc = ws if training else ops.workspace(cfg, True, dev)
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"], Ws,
                  saved=sv, ws=wsc)
    counts = sv["counts"].cpu().numpy()
    out = {"workload": workload_config(ls)["workload"], "value": round(job_throughput(layer_flops(ls, training), ms,
                                                                                      world), 2),
           "unit": "TFLOPS", "ms_per_step": round(ms, 4), "steps": steps,
           "tokens_per_s": round(world * ls.T / (ms * 1e-3), 1), "dtype": "bf16",
           "expert_counts": {"min": int(counts.min()), "max": int(counts.max()), "mean": round(float(counts.mean()), 1),
                             "zero_token_experts": int((counts == 0).sum())},
           "kernels": kernels}
    if ls.skew:
        # the skewed regime's defining property: a dominant expert and
        # experts that receive no token
        assert counts.max() > 8 * counts.mean() and (counts == 0).sum() >= 1, out["expert_counts"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fn, fl_s, desc = oracle_sample(ls, d, args.seed, n_experts=2, n_router_tokens=512, max_rows=256)
        t0 = time.perf_counter()
        fn()
        one = time.perf_counter() - t0
        reps = max(1, min(10, int(3.0 / max(one, 1e-3))))
        tflops, dt = time_oracle(fn, fl_s, reps)
        out["cpu_baseline"] = {"value": round(tflops, 6), "unit": "TFLOPS", "cores": blas_threads(), "kind": "oracle",
                               "sample": desc + f" (at most 256 rows per expert); {reps} repetitions, {dt:.2f} s each"}
    del d, ws, saved, grads, y, sv, wsc
    torch.cuda.empty_cache()
    return out


def gemm_source_sha():
    """sha256 prefix of the GEMM kernel sources (the traffic figures in
    profiles/traffic.json hold only for the sources they were captured on)."""
    import hashlib
    d = os.path.join(ROOT, "route_permute_grouped_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_tc.cuh", "epilogue.cuh", "common.cuh"):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(kernel):
    """DRAM bytes per launch of `kernel` (dram__bytes_read.sum +
    dram__bytes_write.sum) from the committed ncu summary, or None when it was
    not captured or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        ent = json.load(open(p)).get(kernel)
        if ent is None or ent.get("source_sha") != gemm_source_sha():
            return None
        return ent.get("dram_bytes_per_launch")
    except Exception:
        return None


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from route_permute_grouped_gb300 import synth
    ls = synth.shape(args.workload, force_balanced=bool(getattr(args, "force_balanced", False)))
    if getattr(args, "recompute", False):
        ls.extra["recompute"] = True
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, ls)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, ls, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
