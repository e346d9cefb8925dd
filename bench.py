#!/usr/bin/env python
"""Benchmark of the fused MoE expert layer on GB300: forward, backward and the activation-
checkpointed layer (2 x forward + backward), in ms and TFLOP/s, with the fraction of the measured
bf16 tensor peak.

A step is one checkpointed layer over the Qwen3-30B-A3B-shaped workload (T=16384 tokens, H=2048,
I=768, 128 experts, top-8, uniform routing): a forward, a forward that saves [g|u] (the
recompute), and a backward that reuses it.  FLOPs are algorithmic: 2*T*k*H*3I per forward, twice
that per backward; recompute FLOPs are not credited.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded token sample of the same workload (there is
no runnable reference implementation).  Under torchrun each rank runs an independent replica of
the layer (no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd/bwd/2xfwd+bwd ms & TFLOP/s (% of GB300 tensor peak), 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="qwen3_30b_a3b")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-mx", action="store_true", help="skip the MXFP8 measurement of the same layer")
    p.add_argument("--no-extra", action="store_true", help="skip the 235B-shaped and Zipf-routed workloads")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------------------------------ dist
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.6)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as fh:
            rows = [ln.strip().split(", ") for ln in fh if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1])); smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------ ours
# DRAM bytes (read + write) per launch of a kernel, from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of the current build on the profile_30b_e32 workload (4096 tokens, 32
# experts: the 30B layer's per-expert work), scaled x4 to the 128-expert layer, since every size
# grows with E at equal per-expert work.  The forward gate/up figure is its saving launch (344.0 MB
# read, 128.7 MB written; the build whose epilogue stores w h).  A kernel changed since its capture
# is left out (null).
PROFILED_TRAFFIC = {("qwen3_30b_a3b", "gemm_fwd_gate_up_swiglu"): 4 * (343.972e6 + 128.740e6)}

GEMM_FLOPS = {  # algorithmic FLOPs per launch of each grouped GEMM (BF16 or MXFP8), in units of S*H*I
    "gemm_fwd_gate_up_swiglu": 4, "gemm_fwd_gate_up_save": 4, "gemm_fwd_down_weighted": 2,
    "gemm_bwd_down_swiglu_bwd": 2, "gemm_bwd_gate_up": 4, "gemm_wgrad_down": 2, "gemm_wgrad_gate_up": 4,
    "gemm_fwd_down_reduce": 2,
}


def oracle_step(cfg, a, dy):
    """One step of the workload by the oracle in the workload's precision (quantise-dequantise at
    the same points as the layer): 2 x forward + backward, or the forward alone for the
    forward-only FP8 x FP4 layer.  Returns the step's algorithmic FLOPs per token-sample FLOP unit."""
    import oracle
    fwd_kw = {"mxfp8": {"mxfp8": True}, "fp8_fp4": {"fp8_fp4": True}}.get(cfg.precision, {})
    bwd_kw = {"mxfp8": {"mxfp8": True}, "fp8_bwd": {"fp8_bwd": True}}.get(cfg.precision, {})
    oracle.forward(*a, **fwd_kw)
    if cfg.precision == "fp8_fp4":
        return 1
    oracle.forward(*a, **fwd_kw)
    oracle.backward(dy, *a, **bwd_kw)
    return 4


def cpu_baseline(cfg, budget_s: float, seed_tokens: int = 256):
    """The oracle as it stands, on a token sample of the workload (all E experts, same k)."""
    import numpy as np

    from moe_expert_layer_permute_gb300 import inputs as gen
    cores = len(os.sched_getaffinity(0))
    Ts = seed_tokens
    sub = gen.custom_config(name=cfg.name + "_sample", T=Ts, H=cfg.H, I=cfg.I, E=cfg.E, k=cfg.k,
                            routing=cfg.routing, seed=cfg.seed)
    inp = gen.make_inputs(sub)
    args = (inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2"))
    dy = inp.f64("dy")
    runs = []
    t_end = time.time() + budget_s
    while True:
        t0 = time.perf_counter()
        units = oracle_step(cfg, args, dy)
        runs.append(time.perf_counter() - t0)
        if time.time() > t_end or len(runs) >= 3:
            break
    sec = statistics.median(runs)
    flops = units * sub.fwd_flops()
    del np
    what = "forward" if units == 1 else "checkpointed layer 2xfwd+bwd"
    return {"value": flops / sec / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{Ts} tokens of {cfg.name} (all {cfg.E} experts, top-{cfg.k}), fp64 numpy {cfg.precision}, "
                      f"{what}, median of {len(runs)} runs ({sec:.2f} s each)",
            "seconds_per_layer_sample": sec}


def host_tensor(a):
    """A numpy input array as a CPU torch tensor (bf16 bit patterns reinterpreted)."""
    import numpy as np
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def timed(fn, n, ws, stream):
    """Milliseconds of n calls of fn between CUDA events on `stream`, with a barrier and a device
    synchronisation on both sides; the maximum over ranks."""
    import torch
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return allreduce_max(e0.elapsed_time(e1), ws)


def measure(bd, gen, cfg, steps, warmup, ws, local, with_e2e, fwd_flags=0):
    """Times fwd, bwd and the checkpointed layer for one workload; returns a dict of results.
    fwd_flags are OR-ed into every forward call (MOE_FLAG_FUSED_COMBINE for the fused variant)."""
    import torch

    dev = torch.device("cuda", local)
    inp = cached_inputs(gen, cfg)
    h_in = {n: host_tensor(getattr(inp, n)) for n in ("x", "topk_idx", "topk_w", "W13", "W2", "dy")}
    if with_e2e:   # the end-to-end leg copies its per-step inputs from pinned host memory
        h_in = {n: (t.pin_memory() if n not in ("W13", "W2") else t) for n, t in h_in.items()}
    del inp
    d = {n: t.to(dev) for n, t in h_in.items()}
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    mx = cfg.precision == "mxfp8"
    mx_bwd = cfg.precision in ("mxfp8", "fp8_bwd")
    wdt = torch.float32 if mx_bwd else torch.bfloat16  # MXFP8 backward: master weight gradients in fp32
    d["y"] = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    d["dx"] = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    d["dW13"] = torch.empty(E, 2 * I, H, dtype=wdt, device=dev)
    d["dW2"] = torch.empty(E, H, I, dtype=wdt, device=dev)
    d["dtw"] = torch.empty(T, k, dtype=torch.float32, device=dev)
    prec = {"bf16": bd.MOE_BF16, "mxfp8": bd.MOE_MXFP8, "fp8_bwd": bd.MOE_FP8_BWD}[cfg.precision]
    sc = bd.Scratch(T, H, I, E, k, precision=prec, device=dev)
    stream = torch.cuda.current_stream()
    # MXFP8: the first forward of a step quantises the weights, the later calls reuse the copies;
    # fp8_bwd: only the backward quantises them
    RW = bd.MOE_FLAG_REUSE_WEIGHTS if mx else 0

    def fwd(flags=0):
        bd.moe_fwd(d["x"], d["topk_idx"], d["topk_w"], d["W13"], d["W2"], d["y"], sc, flags=flags | fwd_flags)

    def bwd(flags=0):
        bd.moe_bwd(d["dy"], d["x"], d["topk_idx"], d["topk_w"], d["W13"], d["W2"], d["dx"], d["dW13"], d["dW2"],
                   d["dtw"], sc, flags=flags)

    def step():
        # one training step of the checkpointed layer: the weights (and their MXFP8 copies) are
        # made once, the recompute saves [g|u], the backward reuses both; a new step is a new epoch
        # (an optimizer would have updated the weights in place)
        sc.epoch += 1
        fwd()
        fwd(bd.MOE_FLAG_SAVE_GU | RW)
        bwd(bd.MOE_FLAG_REUSE_FWD | RW)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    if bd.moe_read_device_status(sc) != 0:
        raise RuntimeError("device status word set during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    # forward alone (each call makes its own MXFP8 weight copies) and backward alone (reusing a
    # saved forward, as in the layer)
    fwd_ms = timed(fwd, steps, ws, stream) / steps
    fwd(bd.MOE_FLAG_SAVE_GU)
    bwd_ms = timed(lambda: bwd(bd.MOE_FLAG_REUSE_FWD | RW), steps, ws, stream) / steps
    # the checkpointed layer; then the same steps again with per-kernel CUDA events recorded on
    # the launch stream (the events between launches cost time, so they are not in full_ms)
    full_total = timed(step, steps, ws, stream)
    bd.moe_trace_reset()
    bd.moe_trace_enable(True)
    traced_steps = max(3, min(steps, 50))
    timed(step, traced_steps, ws, stream)
    bd.moe_trace_enable(False)
    kern = bd.moe_trace_read()
    clk = clocks.stop()
    full_ms = full_total / steps
    status = bd.moe_read_device_status(sc)
    out = {"cfg": cfg, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "full_ms": full_ms, "kern": kern, "clocks": clk,
           "status": status, "steps": steps, "traced_steps": traced_steps}
    if with_e2e:
        # End to end through the public API with host buffers.  Every step copies its data in from
        # pinned host memory (x, dy and the routing: the layer's per-step inputs) and its results
        # back (y and dx to the neighbouring layers, dtopk_w to the router); the parameters W13, W2
        # stay on the device as in training, where the optimizer consumes dW13, dW2 there.  Steps
        # are pipelined as an input pipeline prefetches: double-buffered device tensors, copies on
        # their own streams, each buffer reused only after the step that read it and the copy-out
        # of its results have finished.
        IN, OUT, NB = ("x", "dy", "topk_idx", "topk_w"), ("y", "dx", "dtw"), 2
        dev_in = [{n: torch.empty_like(d[n]) for n in IN} for _ in range(NB)]
        dev_out = [{n: torch.empty_like(d[n]) for n in OUT} for _ in range(NB)]
        h_out = [{n: torch.empty(d[n].shape, dtype=d[n].dtype).pin_memory() for n in OUT} for _ in range(NB)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(NB)]
        ev_done = [torch.cuda.Event() for _ in range(NB)]
        ev_out = [torch.cuda.Event() for _ in range(NB)]
        h2d = sum(h_in[n].numel() * h_in[n].element_size() for n in IN)
        d2h = sum(h_out[0][n].numel() * h_out[0][n].element_size() for n in OUT)

        def layer_step(bi, bo):
            args = (bi["topk_idx"], bi["topk_w"], d["W13"], d["W2"])
            sc.epoch += 1
            bd.moe_fwd(bi["x"], *args, bo["y"], sc, flags=0)
            bd.moe_fwd(bi["x"], *args, bo["y"], sc, flags=bd.MOE_FLAG_SAVE_GU | RW)
            bd.moe_bwd(bi["dy"], bi["x"], *args, bo["dx"], d["dW13"], d["dW2"], bo["dtw"], sc,
                       flags=bd.MOE_FLAG_REUSE_FWD | RW)

        def e2e_run(n):
            compute = torch.cuda.current_stream()
            s_in.wait_stream(compute)
            s_out.wait_stream(compute)
            for i in range(n):
                b = i % NB
                with torch.cuda.stream(s_in):
                    s_in.wait_event(ev_done[b])          # the step that last read dev_in[b] is done
                    for k_ in IN:
                        dev_in[b][k_].copy_(h_in[k_], non_blocking=True)
                    ev_in[b].record(s_in)
                compute.wait_event(ev_in[b])
                compute.wait_event(ev_out[b])            # dev_out[b]'s previous results are copied out
                layer_step(dev_in[b], dev_out[b])
                ev_done[b].record(compute)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[b])
                    for k_ in OUT:
                        h_out[b][k_].copy_(dev_out[b][k_], non_blocking=True)
                    ev_out[b].record(s_out)
            compute.wait_stream(s_in)
            compute.wait_stream(s_out)

        e2e_steps = max(3, min(steps, 20))
        e2e_run(2)
        out["e2e_ms"] = timed(lambda: e2e_run(e2e_steps), 1, ws, stream) / e2e_steps
        out["h2d"], out["d2h"] = h2d, d2h
        out["e2e_copies"] = ("per step: x, dy, topk_idx, topk_w host->device and y, dx, dtopk_w device->host "
                             "(pinned host memory; W13, W2 resident and dW13, dW2 kept on the device as in "
                             "training); steps pipelined with double-buffered device tensors and copy streams")
    del d, sc
    torch.cuda.empty_cache()
    return out


def fwd_measure(bd, gen, cfg, steps, warmup, ws, local, peak, peak_src):
    """The forward alone in a forward-only precision (FP8 x FP4): per call with the weights
    quantised in the call, and with the copies made once (MOE_FLAG_REUSE_WEIGHTS, fixed weights as
    when serving); per-kernel times of the latter and the roofline of its dominant GEMM."""
    import torch

    dev = torch.device("cuda", local)
    inp = cached_inputs(gen, cfg)
    d = {n: host_tensor(getattr(inp, n)).to(dev) for n in ("x", "topk_idx", "topk_w", "W13", "W2")}
    del inp
    d["y"] = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    prec = {"fp8_fp4": bd.MOE_FP8_FP4, "mxfp8": bd.MOE_MXFP8}[cfg.precision]
    sc = bd.Scratch(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, precision=prec, device=dev)
    stream = torch.cuda.current_stream()
    RW = bd.MOE_FLAG_REUSE_WEIGHTS

    def fwd(flags=0):
        bd.moe_fwd(d["x"], d["topk_idx"], d["topk_w"], d["W13"], d["W2"], d["y"], sc, flags=flags)

    fwd()
    for _ in range(max(3, warmup)):
        fwd(RW)
    torch.cuda.synchronize()
    if bd.moe_read_device_status(sc) != 0:
        raise RuntimeError("device status word set during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    q_ms = timed(fwd, steps, ws, stream) / steps
    r_ms = timed(lambda: fwd(RW), steps, ws, stream) / steps
    bd.moe_trace_reset()
    bd.moe_trace_enable(True)
    traced = max(3, min(steps, 50))
    timed(lambda: fwd(RW), traced, ws, stream)
    bd.moe_trace_enable(False)
    kern = bd.moe_trace_read()
    clk = clocks.stop()
    status = bd.moe_read_device_status(sc)
    del d, sc
    torch.cuda.empty_cache()
    fl = cfg.fwd_flops()
    shf = float(cfg.S) * cfg.H * cfg.I
    total = sum(v[1] for v in kern.values())
    rows = {n: {"launches": c, "avg_ms": ms / c, "share": ms / total if total else None} for n, (c, ms) in kern.items()}
    gemms = {n: v for n, v in rows.items() if n.replace("gemm_mx_", "gemm_") in GEMM_FLOPS}
    top = max(gemms, key=lambda n: gemms[n]["avg_ms"] * gemms[n]["launches"])
    ach = GEMM_FLOPS[top.replace("gemm_mx_", "gemm_")] * shf / (gemms[top]["avg_ms"] * 1e-3) / 1e12
    return {"workload": cfg.name, "fwd_ms": q_ms, "fwd_ms_reuse_weights": r_ms,
            "fwd_tflops": fl / (q_ms * 1e-3) / 1e12, "fwd_tflops_reuse_weights": fl / (r_ms * 1e-3) / 1e12,
            "frac_of_peak_reuse_weights": fl / (r_ms * 1e-3) / 1e12 / peak,
            "peak_tflops": {"value": peak, "source": peak_src},
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "traffic": None, "kernel": top, "peak_source": peak_src},
            "gpu_launches_per_fwd": int(sum(v[0] for v in kern.values()) // traced),
            "kernels": rows, "clocks": clk, "device_status": status}


def router_measure(bd, gen, cfg, reps, hbm_peak):
    """The router before the layer (top-k + softmax over the selected, and its backward) on the
    workload's T x E logits.  One timed iteration is a CUDA graph of NB launches over NB distinct
    buffers (together larger than L2, so no flush is needed and no host launch cost is timed);
    per-launch time = iteration time / NB.  Algorithmic bytes: forward T*E*4 read + T*k*8
    written, backward T*k*12 read + T*E*4 written."""
    import torch
    logits, dtw = gen.router_inputs(cfg)
    T, E, k = cfg.T, cfg.E, cfg.k
    NB = max(2, -(-(256 << 20) // (T * E * 4)))        # >= 256 MiB of logits (and of dlogits)
    lg = [torch.from_numpy(logits).cuda() for _ in range(NB)]
    dw = torch.from_numpy(dtw).cuda()
    idx = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(NB)]
    w = [torch.empty(T, k, dtype=torch.float32, device="cuda") for _ in range(NB)]
    dl = [torch.empty(T, E, dtype=torch.float32, device="cuda") for _ in range(NB)]
    side = torch.cuda.Stream()

    def graph(fn):
        with torch.cuda.stream(side):
            for _ in range(2):
                fn(side)
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                fn(side)
        return g

    g_f = graph(lambda st: [bd.moe_router_fwd(lg[i], idx[i], w[i], stream=st) for i in range(NB)])
    g_b = graph(lambda st: [bd.moe_router_bwd(idx[i], w[i], dw, dl[i], stream=st) for i in range(NB)])
    stream = torch.cuda.current_stream()

    def time_graph(g):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * NB)
    f_ms, b_ms = time_graph(g_f), time_graph(g_b)
    fb, bb = T * E * 4 + T * k * 8, T * k * 12 + T * E * 4
    return {"workload": f"T={T} E={E} k={k} fp32 logits ~ N(0,1)", "fwd_us": f_ms * 1e3, "bwd_us": b_ms * 1e3,
            "fwd_gbs": fb / (f_ms * 1e-3) / 1e9, "bwd_gbs": bb / (b_ms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "peak": hbm_peak, "unit": "GB/s",
                         "fwd_frac": fb / (f_ms * 1e-3) / 1e9 / hbm_peak, "bwd_frac": bb / (b_ms * 1e-3) / 1e9 / hbm_peak},
            "timing": f"CUDA graph of {NB} launches on {NB} distinct buffers (> L2), {reps} replays, per launch",
            "gpu_launches": 2 * NB * reps}


def summarize(m, peak, peak_src):
    """Per-kernel table, dominant-GEMM roofline and layer throughput of one measurement."""
    cfg, kern = m["cfg"], m["kern"]
    fwd_fl = cfg.fwd_flops()
    shf = float(cfg.S) * cfg.H * cfg.I
    total_ms = sum(v[1] for v in kern.values())
    rows = {name: {"launches": n, "avg_ms": ms / n, "share": ms / total_ms if total_ms else None}
            for name, (n, ms) in kern.items()}
    gemms = {n: v for n, v in rows.items() if n.replace("gemm_mx_", "gemm_") in GEMM_FLOPS}
    top = max(gemms, key=lambda n: gemms[n]["avg_ms"] * gemms[n]["launches"]) if gemms else None
    roof = None
    if top:
        ach = GEMM_FLOPS[top.replace("gemm_mx_", "gemm_")] * shf / (gemms[top]["avg_ms"] * 1e-3) / 1e12
        traffic = PROFILED_TRAFFIC.get((cfg.name, top))
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": traffic, "kernel": top, "peak_source": peak_src}
        if traffic is not None:
            roof["traffic_source"] = ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture on "
                                      "profile_30b_e32, x4 to the 128-expert layer (bytes per launch)")
    full_tf = 4 * fwd_fl / (m["full_ms"] * 1e-3) / 1e12
    return {"fwd_ms": m["fwd_ms"], "bwd_ms": m["bwd_ms"], "full_ms": m["full_ms"],
            "fwd_tflops": fwd_fl / (m["fwd_ms"] * 1e-3) / 1e12,
            "bwd_tflops": 2 * fwd_fl / (m["bwd_ms"] * 1e-3) / 1e12,
            "full_tflops": full_tf, "frac_of_peak": full_tf / peak,
            "identity_2fwd_plus_bwd_ms": 2 * m["fwd_ms"] + m["bwd_ms"],
            # launches in the timed steps: the traced launches per step times the timed steps
            "roofline": roof, "gpu_launches": int(sum(v[0] for v in kern.values()) * m["steps"] // m["traced_steps"]),
            "kernels": rows,
            "clocks": m["clocks"], "device_status": m["status"]}


# Workloads measured beside the headline one in the default run, each as its own checkpointed
# layer step: the Qwen3-235B-A22B-shaped layer in BF16 and MXFP8, and Zipf-skewed routing on the
# 30B shape at 16,384 and 4,096 tokens.
EXTRA_WORKLOADS = ("qwen3_235b_a22b", "qwen3_235b_a22b_mxfp8", "skew_zipf_16k", "skew_zipf_4k")


def peak_table(peaks, src):
    """Denominators of the fractions.  The timed regions are short (tens of steps, well under a
    second), so the headline divides by the measured burst bf16 rate; the sustained rate, taken over
    a seconds-long loop at a lower SM clock, is reported beside it."""
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sust = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    sust_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    # MXFP8 at the recipe's nominal dense ratio 4.5 : 2.25; fp8_bwd: two BF16 forwards (2F) and one
    # MXFP8 backward (2F), so its peak is the harmonic blend 4F / (2F / P + 2F / 2P) = 4P / 3
    def by_prec(p):
        return {"bf16": p, "mxfp8": 2.0 * p, "fp8_bwd": 4.0 * p / 3.0, "fp8_fp4": 2.0 * p}
    names = {"bf16": "", "mxfp8": " x 2 (nominal MXFP8:BF16 ratio)",
             "fp8_bwd": " blended with 2x it (BF16 forwards, MXFP8 backward): 4/3 x",
             "fp8_fp4": " x 2 (nominal FP8:BF16 ratio; kind::mxf8f6f4 runs E2M1 at it)"}
    return {"burst": by_prec(burst), "sustained": by_prec(sust), "sustained_mhz": sust_mhz,
            "src": {k: f"{src} bf16_tflops (burst){v}" for k, v in names.items()}}


_INPUT_CACHE = {}


def cached_inputs(gen, cfg):
    """Seeded inputs of a workload; workloads that differ only in precision share them."""
    key = (cfg.seed, cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.routing)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = gen.make_inputs(cfg)
    return _INPUT_CACHE[key]


def secondary_fracs(sm, prec, pk):
    """The full layer's fraction of the sustained peak, with the clocks behind both numbers."""
    return {"frac_of_sustained_peak": sm["full_tflops"] / pk["sustained"][prec],
            "sustained_peak_tflops": pk["sustained"][prec], "sustained_peak_sm_mhz": pk["sustained_mhz"],
            "run_sm_mhz": (sm.get("clocks") or {}).get("sm_mhz")}


def compact(name, sm):
    """One workload's headline numbers (repeated last in the JSON line)."""
    r = {k: round(sm[k], 4) for k in ("fwd_ms", "bwd_ms", "full_ms", "full_tflops", "frac_of_peak") if k in sm}
    if "fwd_ms_reuse_weights" in sm:
        r.update({"fwd_ms_reuse_weights": round(sm["fwd_ms_reuse_weights"], 4),
                  "fwd_tflops_reuse_weights": round(sm["fwd_tflops_reuse_weights"], 1),
                  "frac_of_peak": round(sm["frac_of_peak_reuse_weights"], 4)})
    if sm.get("roofline"):
        r["top_kernel"] = sm["roofline"]["kernel"]
        r["top_kernel_frac"] = round(sm["roofline"]["frac"], 4)
    r["sm_mhz"] = (sm.get("clocks") or {}).get("sm_mhz")
    return r


def run_ours(args, rank, ws, local):
    import torch

    from moe_expert_layer_permute_gb300 import build as b
    b.build()
    from moe_expert_layer_permute_gb300 import binding as bd
    from moe_expert_layer_permute_gb300 import inputs as gen

    torch.cuda.set_device(local)
    cfg = gen.CONFIGS[args.config]
    peaks, src = load_peaks()
    pk = peak_table(peaks, src)
    summary = {}
    if cfg.precision == "fp8_fp4":
        # a forward-only layer: the line is its forward with the weight copies made once
        f4 = fwd_measure(bd, gen, cfg, args.steps, args.warmup, ws, local, pk["burst"]["fp8_fp4"],
                         pk["src"]["fp8_fp4"])
        summary[cfg.name] = compact(cfg.name, f4)
        return {
            "metric": METRIC, "value": f4["fwd_tflops_reuse_weights"] * ws, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": f4["fwd_ms_reuse_weights"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8-e4m3 x mxfp4-e2m1",
            "data": "synthetic: seeded N(0,1) x, N(0,1/sqrt(fan_in)) weights, uniform top-8 routing, softmax weights",
            "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} k={cfg.k} fp8_fp4 "
                                   f"{cfg.routing} routing",
                       "step": "fwd (forward only; weight copies made once)",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "roofline": f4["roofline"], "gpu_launches": f4["gpu_launches_per_fwd"] * args.steps,
            "clocks": f4["clocks"], "device_status": f4["device_status"], "fp8_fp4_fwd": f4, "cpu_baseline": None,
            "summary": summary,
        }
    prec = cfg.precision
    m = measure(bd, gen, cfg, args.steps, args.warmup, ws, local, with_e2e=True)
    sm = summarize(m, pk["burst"][prec], pk["src"][prec])
    line = {
        "metric": METRIC, "value": sm["full_tflops"] * ws, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sm["full_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "mxfp8": "mxfp8-e4m3", "fp8_bwd": "bf16 fwd / mxfp8-e4m3 bwd"}[prec],
        "data": "synthetic: seeded N(0,1) x/dy, N(0,1/sqrt(fan_in)) weights, uniform top-8 routing, softmax weights",
        "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} k={cfg.k} {prec} "
                               f"{cfg.routing} routing",
                   "step": "fwd + fwd(save [g|u]) + bwd(reuse)", "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2 (weights alone 1.13 GiB per step)"},
        "peak_tflops": {"value": pk["burst"][prec], "source": pk["src"][prec]},
    }
    line.update({k: v for k, v in sm.items() if k not in ("clocks", "device_status")})
    line.update(secondary_fracs(sm, prec, pk))
    line["e2e"] = {"value": 4 * cfg.fwd_flops() / (m["e2e_ms"] * 1e-3) / 1e12 * ws, "unit": "TFLOP/s",
                   "ms_per_step": m["e2e_ms"], "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                   "copies": m["e2e_copies"]}
    line["clocks"] = sm["clocks"]
    line["device_status"] = sm["device_status"]
    summary[cfg.name] = compact(cfg.name, sm)

    def side(name, steps, fwd_flags=0, label=None):
        c = gen.CONFIGS[name]
        mm = measure(bd, gen, c, steps, args.warmup, ws, local, with_e2e=False, fwd_flags=fwd_flags)
        r = summarize(mm, pk["burst"][c.precision], pk["src"][c.precision])
        r["workload"] = f"{c.name}: T={c.T} H={c.H} I={c.I} E={c.E} k={c.k} {c.precision} {c.routing} routing"
        r["peak_tflops"] = {"value": pk["burst"][c.precision], "source": pk["src"][c.precision]}
        r.update(secondary_fracs(r, c.precision, pk))
        summary[label or c.name] = compact(c.name, r)
        return r

    if not args.no_extra and prec == "bf16":
        # the combine fused into the down projection (atomic fp32 reduction by token, opt-in flag)
        line["fused_combine"] = side(args.config, args.steps, bd.MOE_FLAG_FUSED_COMBINE,
                                     label=args.config + "_fused_combine")

    if not args.no_mx and prec == "bf16":
        # the same layer in MXFP8 (E4M3 + E8M0 per 32 along K, fp32 weight gradients) and with the
        # BF16 forward and the MXFP8 backward
        for suffix in ("_mxfp8", "_fp8_bwd"):
            if args.config + suffix in gen.CONFIGS:
                line[suffix[1:]] = side(args.config + suffix, args.steps)
        if args.config + "_fp8_fp4" in gen.CONFIGS:
            # the forward-only FP8 x FP4 layer beside the MXFP8 forward, both with weight copies made once
            f4 = fwd_measure(bd, gen, gen.CONFIGS[args.config + "_fp8_fp4"], args.steps, args.warmup, ws, local,
                             pk["burst"]["fp8_fp4"], pk["src"]["fp8_fp4"])
            if args.config + "_mxfp8" in gen.CONFIGS:
                f8 = fwd_measure(bd, gen, gen.CONFIGS[args.config + "_mxfp8"], args.steps, args.warmup, ws, local,
                                 pk["burst"]["mxfp8"], pk["src"]["mxfp8"])
                f4["mxfp8_fwd_ms_reuse_weights"] = f8["fwd_ms_reuse_weights"]
            line["fp8_fp4_fwd"] = f4
            summary[args.config + "_fp8_fp4"] = compact(args.config + "_fp8_fp4", f4)
    if not args.no_extra and args.config == "qwen3_30b_a3b":
        line["workloads"] = {n: side(n, min(args.steps, 20)) for n in EXTRA_WORKLOADS
                             if not (args.no_mx and gen.CONFIGS[n].precision != "bf16")}
    # the router that precedes the layer (outside the layer step, as in the pages' benchmark)
    line["router"] = router_measure(bd, gen, cfg, 20, peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=20.0)
    elif rank == 0:
        line["cpu_baseline"] = None
    summary["router"] = {"fwd_us": round(line["router"]["fwd_us"], 2), "bwd_us": round(line["router"]["bwd_us"], 2)}
    line["summary"] = summary      # last, so that a truncated log keeps every workload's headline
    return line


def run_reference(args, rank, ws):
    """The fp64 oracle timed on the host cores, each step a bounded token sample of the workload."""
    import numpy as np

    from moe_expert_layer_permute_gb300 import inputs as gen
    cfg = gen.CONFIGS[args.config]
    cores = len(os.sched_getaffinity(0))
    Ts = 64
    sub = gen.custom_config(name=cfg.name + "_sample", T=Ts, H=cfg.H, I=cfg.I, E=cfg.E, k=cfg.k,
                            routing=cfg.routing, seed=cfg.seed)
    inp = gen.make_inputs(sub)
    a = (inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2"))
    dy = inp.f64("dy")
    fwd_only = cfg.precision == "fp8_fp4"

    units = 1 if fwd_only else 4
    for _ in range(args.warmup):
        oracle_step(cfg, a, dy)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(cfg, a, dy)
    sec = (time.perf_counter() - t0) / args.steps
    val = units * sub.fwd_flops() / sec / 1e12
    del np
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same recipe as ours)",
            "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} k={cfg.k} "
                                   f"{cfg.precision} {cfg.routing} routing",
                       "step": "fwd (oracle)" if fwd_only else "fwd + fwd + bwd (oracle)",
                       "parallelism": "single process"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{Ts} tokens of {cfg.name} per step (all {cfg.E} experts, top-{cfg.k}), "
                                       f"fp64 numpy {'forward' if fwd_only else 'checkpointed layer'}"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, ws)), flush=True)
        return
    line = run_ours(args, rank, ws, local)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
