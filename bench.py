#!/usr/bin/env python
"""Benchmark of the MoE layer forward + backward on GB300.

One step = one forward and one backward pass of the whole layer (router,
top-k, dispatch tables, permute, fc1 + SwiGLU, fc2, combine; gate gradient,
fc2 dgrad + SwiGLU backward, fc2 wgrad, fc1 dgrad, fc1 wgrad, router
backward, unpermute-reduce) through the C ABI, on seeded synthetic inputs of
the DeepSeek-V3-shaped expert layer by default (T=8192, H=7168, 256 routed
experts, top-8 sigmoid routing with a per-expert logit bias, SwiGLU F=2048,
plus one shared expert with F=2048, bf16: the largest of the workloads that
fit one GPU); --workload selects the Mixtral-8x7B- and Qwen3-235B-shaped
layers and the blockwise-FP8 variant. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores on a bounded
token sample of the same workload (the layer has no runnable reference
implementation). Multi-GPU runs are independent replicas (weak scaling):
every rank runs its own layer and the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer fwd+bwd TFLOPS and % of GB300 tensor peak; tokens/s per layer"
GEMM_STAGES = ("fc1_swiglu", "fc2", "fc2_dgrad_swiglu", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad",
               "shared_fc1_swiglu", "shared_fc2", "shared_fc2_dgrad", "shared_fc2_wgrad",
               "shared_fc1_dgrad", "shared_fc1_wgrad")


def stage_flops(name: str, w: mi.Workload) -> float:
    """Algorithmic FLOPs of one launch of a grouped-GEMM stage (2 per MAC,
    routed rows R = T k; zero padding rows not counted)."""
    rows, F = (w.T, w.Fs) if name.startswith("shared_") else (w.R, w.F)
    base = name[len("shared_"):] if name.startswith("shared_") else name
    per = 2.0 * rows * w.H * F
    return {"fc1_swiglu": 2 * per, "fc2": per, "fc2_dgrad_swiglu": per, "fc2_dgrad": per,
            "fc2_wgrad": per, "fc1_dgrad": 2 * per, "fc1_wgrad": 2 * per}[base]


def stage_bytes(name: str, w: mi.Workload) -> float:
    """Algorithmic DRAM bytes of one launch of a grouped-GEMM stage: each
    operand read once and each output written once (routed rows R = T k, no
    padding rows). Operands are E4M3 codes (1 byte, plus one fp32 scale per
    128 elements) in the blockwise FP8 layer, E4M3 codes plus one scale byte
    per 32 in MXFP8, E2M1 codes (half a byte) plus one scale byte per 16 in
    NVFP4, and bf16 otherwise; stored outputs are bf16 (fp32 in the fp32
    layer)."""
    shared = name.startswith("shared_")
    base = name[len("shared_"):] if shared else name
    rows, E, F = (w.T, 1, w.Fs) if shared else (w.R, w.E, w.F)
    H = w.H
    o = 4 if w.dtype == mi.FP32 else 2
    a = 4 if w.dtype == mi.FP32 else (1 + 4 / 128 if w.dtype == mi.FP8_BLOCK else
                                      1 + 1 / 32 if w.dtype == mi.MXFP8 else
                                      0.5 + 1 / 16 if w.dtype == mi.NVFP4 else 2)
    RH, RF, EHF = rows * H, rows * F, E * H * F
    return {"fc1_swiglu": a * (RH + 2 * EHF) + o * 3 * RF,
            "fc2": a * (RF + EHF) + o * RH,
            "fc2_dgrad_swiglu": a * (RH + EHF) + o * 2 * RF + o * 2 * RF,
            "fc2_dgrad": a * (RH + EHF) + o * 2 * RF + o * 2 * RF,
            "fc2_wgrad": a * (RF + RH) + o * EHF,
            "fc1_dgrad": a * (2 * RF + 2 * EHF) + o * RH,
            "fc1_wgrad": a * (RH + 2 * RF) + o * 2 * EHF}[base]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def choose_peak(peaks, kind, clocks, fp8, fp4=False):
    """Tensor peak for this run's clocks: the burst cuBLAS figure unless the
    run's median SM clock is within 5% of the clock the sustained figure was
    measured at (a power-capped, seconds-long loop). FP8 takes twice the bf16
    figure (nominal 4.5 vs 2.25 PFLOP/s dense), FP4 six times (nominal 13.5).
    Returns (peak, description)."""
    burst = peaks["bf16_tflops"]
    sust = peaks.get("bf16_tflops_sustained", burst)
    sust_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    med = clocks.get("sm_mhz")
    if sust_mhz and med and med <= 1.05 * sust_mhz:
        peak, desc = sust, (f"bf16_tflops_sustained of {kind} peaks (measured at a median "
                            f"{sust_mhz:.0f} MHz; this run's median SM clock {med:.0f} MHz)")
    else:
        peak, desc = burst, (f"bf16_tflops (burst) of {kind} peaks (this run's median SM clock "
                             f"{med if med is None else round(med)} MHz is above the "
                             f"{sust_mhz} MHz of the sustained measurement)")
    if fp4:
        peak, desc = 6.0 * peak, "6 x " + desc + " (nominal fp4/bf16 ratio)"
    elif fp8:
        peak, desc = 2.0 * peak, "2 x " + desc + " (nominal fp8/bf16 ratio)"
    return peak, desc


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        if line.startswith("traffic_bytes_per_launch:"):
            v = line.split(":", 1)[1].strip()
            return None if v in ("", "null") else float(v)
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 200 ms."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.p = None

    def _read(self):
        for line in self.p.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self, t0, t1):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        rows = [r for t, r in self.rows if t0 <= t <= t1 and len(r) >= 10]
        window = "timed region"
        if len(rows) < 3:
            rows = [r for _, r in self.rows if len(r) >= 10]
            window = "warm-up and timed region (timed region shorter than 3 samples)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window": window}


# ------------------------------------------------------- multi-rank logic
def reduce_max(v: float, device=None) -> float:
    """Maximum of a per-rank value over all ranks (no-op without a process
    group). Replicas share nothing else: every rank runs its own layer."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_metrics(world: int, ms_per_step_max: float, flops_per_step: float, tokens_per_step: int):
    """Whole-job throughput of `world` replicas timed by the slowest rank."""
    s = ms_per_step_max * 1e-3
    return {"tflops": world * flops_per_step / s / 1e12, "tokens_per_s": world * tokens_per_step / s}


# ---------------------------------------------------------------- oracle leg
def oracle_sample(w: mi.Workload, d, n_tok: int):
    """Time the fp64 oracle (route + forward + backward) on the first n_tok
    tokens of the workload. The sample routes with the full router; its
    expert computation gets only the experts those tokens selected (numbered
    0.. in index order), which is the same arithmetic for those tokens:
    experts that receive no token add nothing to y and dX and have zero
    weight gradients. Returns (seconds, flops of that sample, threads)."""
    import numpy as np
    import oracle
    oracle.build()
    x, dY = d["x"][:n_tok], d["dY"][:n_tok]
    t0 = time.perf_counter()
    r = oracle.route(x, d["Wr"], d["b"], w.k, w.score)
    need = sorted(set(r["topk"].ravel().tolist()))
    renum = np.full(w.E, -1, np.int32)
    renum[need] = np.arange(len(need), dtype=np.int32)
    topk = renum[r["topk"]]
    Wg, Wu, Wd = (np.ascontiguousarray(d[n][need]) for n in ("Wg", "Wu", "Wd"))
    oracle.forward(x, Wg, Wu, Wd, topk, r["gates"], d["Wsg"], d["Wsu"], d["Wsd"])
    oracle.backward(x, np.ascontiguousarray(d["Wr"][:, need]), Wg, Wu, Wd, topk, r["gates"],
                    np.ascontiguousarray(r["scores"][:, need]), dY, w.score, d["Wsg"], d["Wsu"], d["Wsd"])
    dt = time.perf_counter() - t0
    ws = mi.scaled(w, T=n_tok)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return dt, ws.flops_fwd_bwd(), threads


def oracle_host_inputs(inp):
    """fp64 host copies of the inputs for the oracle; the expert weights stay
    in their storage dtype (bf16 or fp32) until a sample picks its experts."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif k in ("Wg", "Wu", "Wd"):
            out[k] = _LazyF64(v.cpu())
        else:
            out[k] = v.cpu().double().numpy()
    return out


class _LazyF64:
    """Expert-stacked weights converted to fp64 only for the experts indexed."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        import torch
        return self.t[torch.as_tensor(idx, dtype=torch.long)].double().numpy()


def host_inputs(w: mi.Workload, device):
    """Seeded inputs generated on `device`, returned on the host."""
    g = mi.make_inputs(w, device)
    return {k: (None if v is None else v.cpu()) for k, v in g.items()}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = oracle_host_inputs(host_inputs(w, dev))
    n_tok = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(w, inp, n_tok)
    total_s, total_f, threads = 0.0, 0.0, 1
    for _ in range(args.steps):
        dt, fl, threads = oracle_sample(w, inp, n_tok)
        total_s += dt
        total_f += fl
    value = total_f / total_s / 1e12
    sample = (f"first {n_tok} tokens of {w.name} (the experts they select); fp64 oracle "
              f"route+forward+backward per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "tokens_per_s": n_tok * args.steps / total_s,
            "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "top_k": w.k, "F": w.F,
                       "Fs": w.Fs, "score": "sigmoid" if w.score else "softmax", "sample_tokens": n_tok},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg
def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from mixture_experts_layer_sigmoid_gb300 import (MoELayer, MOE_BF16, MOE_FP32, MOE_FP8_BLOCK, MOE_MXFP8,
                                                     MOE_NVFP4)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    inp = mi.make_inputs(w, dev)
    layer = MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score,
                     dtype={mi.FP32: MOE_FP32, mi.BF16: MOE_BF16, mi.FP8_BLOCK: MOE_FP8_BLOCK,
                            mi.MXFP8: MOE_MXFP8, mi.NVFP4: MOE_NVFP4}[w.dtype],
                     Fs=w.Fs, device=local, stage_timing=True, fold_gates=args.fold_gates)
    x, dY = inp["x"], inp["dY"]
    W = (inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], inp["Wsg"], inp["Wsu"], inp["Wsd"])
    y = torch.empty_like(x)
    grads = dict(dX=torch.empty_like(x), dWr=torch.empty_like(inp["Wr"]), dW_gate=torch.empty_like(inp["Wg"]),
                 dW_up=torch.empty_like(inp["Wu"]), dW_down=torch.empty_like(inp["Wd"]))
    if w.Fs:
        grads.update(dWs_gate=torch.empty_like(inp["Wsg"]), dWs_up=torch.empty_like(inp["Wsu"]),
                     dWs_down=torch.empty_like(inp["Wsd"]))

    # --weight-cache (FP8 layers): the expert weights are quantised once, before
    # the timed region, as a trainer does once per optimizer step; the step
    # then reads their E4M3 codes from the cache
    cache = layer.quantize_weights(W[1], W[2], W[3]) if args.weight_cache else None
    Wexp = (None, None, None) if cache is not None else (W[1], W[2], W[3])

    def step(xx, dd, yy=None, dXX=None):
        layer.forward(xx, W[0], inp["b"], *Wexp, W[4], W[5], W[6], y=y if yy is None else yy,
                      weight_cache=cache)
        layer.backward(dd, xx, W[0], *Wexp, W[4], W[5], W[6],
                       grads=grads if dXX is None else dict(grads, dX=dXX), weight_cache=cache)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        return reduce_max(v, dev)

    # ---- device-timed region (inputs resident in HBM)
    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step(x, dY)
    torch.cuda.synchronize()
    if layer.status(w.T) != 0:
        raise RuntimeError("device status word reports an error after warm-up")
    layer.stage_times()                      # clear the warm-up record
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step(x, dY)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    ms = max_over_ranks(e0.elapsed_time(e1)) / args.steps
    stages = layer.stage_times()
    if layer.status(w.T) != 0:
        raise RuntimeError("device status word reports an error in the timed region")

    # ---- end to end through the C ABI with host buffers. Every step copies
    # its x and dY from pinned host memory and its y and dX back; the copies
    # run on two more streams (host->device, device->host) into double-buffered
    # device tensors, so step i's transfers overlap steps i-1 and i+1 (a
    # prefetching input pipeline), and the timed region ends after the last
    # step's outputs reach the host.
    x_h = x.cpu().pin_memory()
    dY_h = dY.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    dX_h = torch.empty_like(x_h).pin_memory()
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    xb = [torch.empty_like(x) for _ in range(2)]
    db = [torch.empty_like(dY) for _ in range(2)]
    yb = [torch.empty_like(x) for _ in range(2)]
    gb = [torch.empty_like(x) for _ in range(2)]
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "out")}
    e2e_steps = max(1, args.steps)

    def e2e_run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(cs_in):
                if i >= 2:
                    cs_in.wait_event(ev["done"][b])     # step i-2 no longer reads xb/db[b]
                xb[b].copy_(x_h, non_blocking=True)
                db[b].copy_(dY_h, non_blocking=True)
                ev["in"][b].record(cs_in)
            stream.wait_event(ev["in"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])         # step i-2's outputs have left yb/gb[b]
            step(xb[b], db[b], yb[b], gb[b])
            ev["done"][b].record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev["done"][b])
                y_h.copy_(yb[b], non_blocking=True)
                dX_h.copy_(gb[b], non_blocking=True)
                ev["out"][b].record(cs_out)
        stream.wait_stream(cs_in)
        stream.wait_stream(cs_out)

    e2e_run(2)
    torch.cuda.synchronize()
    layer.stage_times()
    barrier()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_run(e2e_steps)
    f1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1)) / e2e_steps
    layer.stage_times()

    flops = w.flops_fwd_bwd()
    jm = job_metrics(world, ms, flops, w.T)
    value = jm["tflops"]
    peaks, peaks_kind = load_peaks()
    peak_sust, peak_name = choose_peak(peaks, peaks_kind, clocks, w.dtype in (mi.FP8_BLOCK, mi.MXFP8),
                                       w.dtype == mi.NVFP4)

    # ---- roofline of the dominant kernel (largest device time in the timed
    # region): the slower of its FLOPs at the tensor peak and its algorithmic
    # bytes at the measured HBM copy bandwidth
    hbm = peaks["hbm_gbs"]
    gemms = {n: v for n, v in stages.items() if n in GEMM_STAGES}

    def bound_ms(n):
        return max(stage_flops(n, w) / (peak_sust * 1e12), stage_bytes(n, w) / (hbm * 1e9)) * 1e3

    # One GEMM stage runs once per step as one launch, or two (CTA pairs over
    # the multi-tile experts, then single CTAs over the one-tile experts):
    # its work and its device time are per step either way.
    dom = max(gemms, key=lambda n: gemms[n][1])
    launches, tot_ms = gemms[dom]
    t_launch = tot_ms / args.steps * 1e-3
    tensor_bound = stage_flops(dom, w) / (peak_sust * 1e12) >= stage_bytes(dom, w) / (hbm * 1e9)
    if tensor_bound:
        achieved, peak, unit = stage_flops(dom, w) / t_launch / 1e12, peak_sust, "TFLOP/s"
    else:
        achieved, peak, unit = stage_bytes(dom, w) / t_launch / 1e9, hbm, "GB/s"
    # Wall time of the GEMMs: the step minus every other stage (the GEMM
    # stages' own times plus the gaps between launches)
    gemm_ms = ms - sum(v[1] for n, v in stages.items() if n not in GEMM_STAGES) / args.steps
    gemm_flops = sum(stage_flops(n, w) for n in gemms)
    gemm_bound_ms = sum(bound_ms(n) for n in gemms)
    roofline = {"kernel": dom, "bound": "tensor" if tensor_bound else "hbm", "achieved": achieved,
                "peak": peak, "unit": unit, "frac": achieved / peak,
                "peak_source": peak_name if tensor_bound else f"hbm_gbs of {peaks_kind} peaks",
                "flops_per_launch": stage_flops(dom, w), "bytes_per_launch": stage_bytes(dom, w),
                "tensor_frac": stage_flops(dom, w) / t_launch / 1e12 / peak_sust,
                "traffic": profiled_traffic(dom, w.name),
                "all_grouped_gemms": {"achieved_tflops": gemm_flops / (gemm_ms * 1e-3) / 1e12,
                                      "tensor_frac": gemm_flops / (gemm_ms * 1e-3) / 1e12 / peak_sust,
                                      "roofline_frac": gemm_bound_ms / gemm_ms,
                                      "share_of_step": gemm_ms / ms,
                                      "wall_ms": gemm_ms},
                "per_gemm": {n: {"ms": v[1] / args.steps, "launches": v[0] / args.steps,
                                 "roofline_ms": bound_ms(n),
                                 "bound": "tensor" if stage_flops(n, w) / (peak_sust * 1e12) >=
                                 stage_bytes(n, w) / (hbm * 1e9) else "hbm",
                                 "frac": bound_ms(n) / (v[1] / args.steps)} for n, v in gemms.items()}}
    per_stage = {n: {"launches_per_step": v[0] / args.steps, "ms_per_step": v[1] / args.steps}
                 for n, v in stages.items()}
    launches_total = sum(v[0] for v in stages.values())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_h = oracle_host_inputs(inp)
        del layer
        dt, fl, threads = oracle_sample(w, inp_h, args.cpu_tokens)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"first {args.cpu_tokens} tokens of {w.name} (the experts they select); "
                         f"fp64 oracle route+forward+backward took {dt:.1f} s. The sample is kept to "
                         f"tens of seconds of host work: the oracle runs near "
                         f"{args.cpu_tokens / dt:.2f} tokens/s, so a 256-token slice would take "
                         f"{256 * dt / args.cpu_tokens / 60:.0f} min",
               "tokens_per_s": args.cpu_tokens / dt}

    if rank == 0:
        es = 4 if w.dtype == mi.FP32 else 2   # weights are passed in bf16 for FP8 too
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": {mi.BF16: "bf16", mi.FP32: "f32", mi.FP8_BLOCK: "e4m3", mi.MXFP8: "e4m3",
                          mi.NVFP4: "e2m1"}[w.dtype],
                "data": "synthetic",
                "tokens_per_s": jm["tokens_per_s"],
                "pct_of_tensor_peak": 100.0 * value / world / peak_sust,
                "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "top_k": w.k, "F": w.F,
                           "Fs": w.Fs, "score": "sigmoid" if w.score else "softmax",
                           "routing_bias": w.bias, "seed": w.seed,
                           "l2": "inputs larger than L2 (expert weights %.2f GB), no flush" %
                                 ((3 * w.E * w.H * w.F + 3 * w.H * w.Fs) * es / 1e9),
                           "parallelism": f"replicas x{world}",
                           "fold_gates": bool(args.fold_gates),
                           "weight_cache": bool(args.weight_cache)},
                "roofline": roofline,
                "cpu_baseline": cpu,
                "e2e": {"value": job_metrics(world, ms_e2e, flops, w.T)["tflops"], "unit": "TFLOP/s",
                        "h2d_bytes_per_step": 2 * x.numel() * x.element_size(),
                        "d2h_bytes_per_step": 2 * x.numel() * x.element_size(),
                        "copies": "pinned host <-> device on two copy streams, double-buffered, "
                                  "overlapping the neighbouring steps"},
                "gpu_launches": launches_total,
                "clocks": clocks,
                "stages": per_stage}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="deepseek_v3", choices=sorted(mi.WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=8, help="oracle sample for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=2, help="oracle sample per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fold-gates", action="store_true",
                    help="memory-efficient permutation: routing weights folded into h")
    ap.add_argument("--weight-cache", action="store_true",
                    help="FP8 layers: quantise the expert weights once, outside the timed steps")
    ap.add_argument("--override", default="",
                    help="comma-separated shape overrides, e.g. F=4096,T=2048 (profiling runs)")
    args = ap.parse_args()
    w = mi.WORKLOADS[args.workload]
    if args.weight_cache and w.dtype not in (mi.FP8_BLOCK, mi.MXFP8, mi.NVFP4):
        ap.error("--weight-cache applies to the FP8 workloads only")
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        w = mi.scaled(w, **{k: int(v) for k, v in kv.items()},
                      name=w.name + "[" + args.override + "]")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
