"""Benchmark of the routed MoE layer on GB300: one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The headline step is one forward + backward pass of the whole layer over the
largest single-GPU workload: a 64K-token slice of a 1M-token sequence (T =
65536, d = 4096, 384 routed experts top-6 + 1 shared, I = 2048, bf16 with
fp32 accumulation and fp32 weight gradients, 30 % vision tokens with their
own routing bias, Zipf(1.1) expert load, g|u recomputed in the backward).
Inputs are seeded synthetic tensors made on the device; they are resident in
HBM when the timed region starts.  The line also carries the same step end to
end from host memory (moe_layer_step_host), the full-width T = 4096 forward,
the T = 8192 forward + backward, the skewed multimodal forward (top-k and
hash routers) and the MXFP8 forward.  N > 1 runs N independent replicas (one
per GPU), since the single-GPU layer has no exchange step: value = all
ranks' tokens / max time.

--impl reference times the CPU oracle (the plain fp64 implementation the
tests compare against) on the host cores, on a bounded sample of tokens of
the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MoE layer tokens/s (fwd, fwd+bwd) at 1 GB300; grouped-GEMM % of BF16 tensor peak")
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (read + write) per algorithmic byte of expert GEMM 1, from an ncu
# capture of the current kernel on a small case of the same workload
# (T=640, E=64: 2.262 GB measured for 2.236 GB algorithmic); traffic grows in
# proportion to the experts streamed, so a full launch is this ratio times its
# algorithmic bytes.
GEMM1_DRAM_PER_ALGORITHMIC_BYTE = 1.0116
# DRAM bytes (read + write) per launch of each grouped-GEMM kernel at the
# 64K-token slice, averaged over the kernel's launches in one step: one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum, one pass) of the
# current kernels, command and per-launch figures in
# profiles/dram_traffic_long_slice_fwd_bwd.md.
LONG_SLICE_DRAM_BYTES_PER_LAUNCH = {
    "expert GEMM 1": (21.61e9 + 30.63e9) / 2,   # forward; recompute (saves g|u)
    "weight gradients": (19.92e9 + 41.26e9) / 2,  # dW2; dW13
    "dgrad 1": 23.99e9,
    "dgrad 2": 24.07e9,
    "expert GEMM 2": 12.06e9,
}
FALLBACK_BF16_TFLOPS = 1900.0
# library kernels of one forward: routing (one fused gate + route kernel, or the
# gate GEMM and the routing kernel), rank, scan, scatter, gather, GEMM1, GEMM2,
# combine
def fwd_launches(fused_route):
    return 8 if fused_route else 9


BWD_LAUNCHES = 9      # gather dY, dgrad2, wgrad2, dgrad1, wgrad1, router bwd, dX, dW_g (2)
BWD_RECOMPUTE_EXTRA = 2


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get(
            "bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------- multi-rank

def dist_barrier(world):
    if world > 1:
        torch.distributed.barrier()


def dist_max(value, world, device="cuda"):
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank, max_ms_per_step):
    """Whole-job tokens/s of N independent replicas timed by the slowest one."""
    return world * tokens_per_rank / (max_ms_per_step / 1e3)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------- workloads

def layer_inputs(wl, device, weights=None):
    from moe_expert_layer_04_gb300 import workloads as W
    inp = W.make_inputs(wl, device=device, with_weights=weights is None)
    if weights is not None:
        inp.update(weights)
    return inp


def fwd_algorithmic_bytes(D, counts):
    """Minimum HBM bytes of the expert GEMMs for one forward: every expert
    with at least one row streams its weights once; activations read/written
    once (x_perm rows in, h out for GEMM 1; h in, y_perm out for GEMM 2)."""
    used = int((counts > 0).sum()) + 1          # + the shared expert
    w13 = used * 2 * D.I * D.d * 2
    w2 = used * D.d * D.I * 2
    g1 = w13 + D.R * D.d * 2 + D.R * D.I * 2
    g2 = w2 + D.R * D.I * 2 + D.R * D.d * 2
    return g1, g2


def mx_fwd_bytes(D, counts):
    """The same minimum bytes for the MXFP8 forward: one byte per operand
    element plus one scale byte per 32 (weights, x_perm, h); y_perm stays
    bf16.  Returns (GEMM 1, GEMM 2, dispatch)."""
    used = int((counts > 0).sum()) + 1
    c = 1 + 1 / 32
    g1 = used * 2 * D.I * D.d * c + D.R * D.d * c + D.R * D.I * c
    g2 = used * D.d * D.I * c + D.R * D.I * c + D.R * D.d * 2
    perm = D.T * D.d * 2 + D.R * D.d * c + D.S * 4 * 6
    return int(g1), int(g2), int(perm)


def fwd_flops(D):
    return 2 * D.T * D.d * D.E + 6 * D.R * D.d * D.I


def workload(args):
    """The named workload, optionally shrunk (--tokens / --experts) for
    profiling captures that must stay a few GB."""
    from moe_expert_layer_04_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    over = {}
    if args.tokens:
        over["T"] = args.tokens
    if args.experts:
        over["E"] = args.experts
    if over:
        wl = W.scaled(wl, name=wl.name + "-" + "-".join(f"{k}{v}" for k, v in over.items()), **over)
    return wl


# ------------------------------------------------------------------- ours

def route_kwargs(inp, mode):
    from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH
    if mode == MOE_ROUTE_HASH:
        return dict(logit_offset=None, mode=mode, input_ids=inp["input_ids"],
                    tid2eid=inp["tid2eid"])
    return dict(logit_offset=inp["logit_offset"])


def forward_breakdown(layer, inp, steps, warmup, mode=0, world=1):
    """Times `steps` forward passes, with CUDA events on the launching stream
    around each of the layer's calls.  Returns (per-call ms, ms per step)."""
    stream = torch.cuda.current_stream()
    rk = route_kwargs(inp, mode)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        layer.route(inp["x"], inp["bias"], inp["is_vision"], **rk)
        if evs is not None:
            evs[1].record(stream)
        layer.dispatch(inp["x"])
        if evs is not None:
            evs[2].record(stream)
        layer.expert_gemm1()
        if evs is not None:
            evs[3].record(stream)
        layer.expert_gemm2()
        if evs is not None:
            evs[4].record(stream)
        layer.combine()
        if evs is not None:
            evs[5].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    ms = dist_max(t0.elapsed_time(t1), world)
    names = ["route", "permute", "expert_gemm1", "expert_gemm2", "combine"]
    per = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
           for j, n in enumerate(names)}
    return per, ms / steps


def kernel_metrics(D, counts, per, hbm, bf16, save_gu=False, fused_route=True, mx=False):
    """Per-call achieved GB/s (algorithmic bytes) and TFLOP/s with their
    fractions of the measured peaks.  Routing reads x and W_g and writes the
    logits (the two-kernel path reads them back once more), ids, weights and
    selected scores.  mx: the MXFP8 forward's bytes, and its expert matmuls
    against the fp8 tensor peak: the measured bf16 peak times the nominal
    fp8 / bf16 ratio of 2 (4.5 / 2.25 PFLOP/s dense)."""
    g1_bytes, g2_bytes = fwd_algorithmic_bytes(D, counts)
    perm_bytes = D.T * D.d * 2 + D.R * D.d * 2 + D.S * 4 * 6
    peak_of = {}
    if mx:
        g1_bytes, g2_bytes, perm_bytes = mx_fwd_bytes(D, counts)
        peak_of = {"expert_gemm1": 2 * bf16, "expert_gemm2": 2 * bf16}
    if save_gu:
        g1_bytes += D.R * 2 * D.I * 4
    g1_flops = 4 * D.R * D.d * D.I
    g2_flops = 2 * D.R * D.I * D.d
    comb_bytes = D.R * D.d * 2 + D.T * D.d * 2 + D.S * 4
    route_bytes = (D.T * D.d * 2 + D.E * D.d * 2 + D.T * D.E * 4 * (1 if fused_route else 2)
                   + D.T * D.k * 12)
    out = {}
    for name, by, fl in (("route", route_bytes, 2 * D.T * D.d * D.E), ("permute", perm_bytes, 0),
                         ("expert_gemm1", g1_bytes, g1_flops), ("expert_gemm2", g2_bytes, g2_flops),
                         ("combine", comb_bytes, 0)):
        sec = per[name] / 1e3
        m = {"ms": round(per[name], 4), "gbs": round(by / sec / 1e9, 1),
             "hbm_frac": round(by / sec / 1e9 / hbm, 4)}
        if fl:
            pk = peak_of.get(name, bf16)
            m["tflops"] = round(fl / sec / 1e12, 1)
            m["tensor_frac"] = round(fl / sec / 1e12 / pk, 4)
            if name in peak_of:
                m["tensor_peak"] = "fp8 (2 x measured bf16)"
        out[name] = m
    gemm_peak = 2 * bf16 if mx else bf16
    roof_ms = max(2 * D.T * D.d * D.E / (bf16 * 1e12) + 6 * D.R * D.d * D.I / (gemm_peak * 1e12),
                  (g1_bytes + g2_bytes + perm_bytes + comb_bytes + route_bytes) / (hbm * 1e9)) * 1e3
    return out, g1_bytes, roof_ms


def run_ours(args, rank, world, local_rank):
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    _lib.load()
    hbm, bf16, bf16_sus, peak_src = peaks()
    # the full-width expert weights (same seed and shapes for every full-width
    # workload)
    weights = {k: v for k, v in layer_inputs(W.WORKLOADS["full_fwd"], dev).items()
               if k in ("W_g", "W13", "W2")}

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    h = run_headline(args, weights, dev, world, hbm, bf16_sus)
    e2e = run_headline_e2e(args, h, world)
    wl, D = h["wl"], h["D"]
    ms_step = h["ms_step"]
    value = replica_throughput(world, D.T, ms_step)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_fwd_bwd(h["inp"], wl, args.cpu_tokens, args.cpu_rows)
    counts = h["counts"]
    kernels, roofline = h["kernels"], h["roofline"]
    layer_roof_ms, alg_flops, launches = h["layer_roof_ms"], h["alg_flops"], h["launches"]
    del h
    torch.cuda.empty_cache()

    full = fb = extra = mx = mxs = None
    if not args.no_extra and not args.tokens and not args.experts:
        full = run_full_fwd(args, weights, dev, world, hbm, bf16, peak_src)
        if not args.no_bwd:
            fb = run_fwd_bwd(args, weights, dev, world)
        extra = run_extra_workloads(args, weights, dev, world, hbm, bf16)
        if not args.no_mx:
            mx = run_mx(args, weights, dev, world, hbm, bf16, ["full_fwd", HEADLINE])
            if full is not None and "full_fwd" in mx:
                mx["full_fwd"]["speedup_vs_bf16"] = round(
                    full["ms_per_step"] / mx["full_fwd"]["ms_per_step"], 3)
            if not args.no_bwd:
                mxs = run_mx_fwd_bwd(args, weights, dev, world, hbm, bf16_sus)
                mxs["speedup_vs_bf16"] = round(ms_step / mxs["ms_per_step"], 3)
    clk = clocks.stop()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {"workload": workload_string(wl),
                   "global_batch": wl.T * world, "seq_len": wl.T,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (%.1f GB of expert weights, %.1f GB of fp32 "
                         "weight gradients per step)" % (3 * (D.E + 1) * D.d * D.I * 2 / 1e9,
                                                         3 * (D.E + 1) * D.d * D.I * 4 / 1e9)},
        "roofline": roofline,
        "layer_roofline_ms": round(layer_roof_ms, 4),
        "layer_roofline_frac": round(layer_roof_ms / ms_step, 4),
        "layer_roofline_basis": "algorithmic FLOPs of forward + backward (%.1f TFLOP, the "
                                "recompute not counted) at the sustained bf16 peak" % (
                                    alg_flops / 1e12),
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "expert_load": {"experts_with_tokens": int((counts > 0).sum()),
                        "min_rows": int(counts.min()), "max_rows": int(counts.max())},
        "full_fwd": full,
        "fwd_bwd": fb,
        "extra_workloads": extra,
        "mx_fwd": mx,
        "mx_fwd_bwd": mxs,
    }
    return line


def workload_string(wl):
    return (f"{wl.name}: forward+backward, T={wl.T} d={wl.d} E={wl.E} routed top-{wl.k} + 1 "
            f"shared, I={wl.I}, scaling {wl.rho}, clamp {wl.clamp}, "
            f"{round(100 * wl.vision_frac)}% vision tokens, Zipf({wl.zipf_s}) expert load, "
            f"fp32 weight gradients" + (", g|u recomputed in the backward" if wl.recompute else ""))


def run_full_fwd(args, weights, dev, world, hbm, bf16, peak_src):
    """The full-width forward (T = 4096, near-uniform load): per-call
    breakdown, the weight-streaming roofline of expert GEMM 1, the forward
    through HostPipeline, the literal-bias variant and one launch vs two for
    the expert matmuls."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import Dims, HostPipeline, MoELayer, ffn_fused_supported
    wl = W.WORKLOADS["full_fwd"]
    D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
    inp = layer_inputs(wl, dev, weights=weights)
    layer = MoELayer(D, weights, wl.rho, wl.clamp)
    stream = torch.cuda.current_stream()
    forward_breakdown(layer, inp, 1, args.warmup)
    counts = layer.counts.cpu().numpy()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    per, ms_step = forward_breakdown(layer, inp, args.steps, 1, world=world)
    kernels, g1_bytes, layer_roof_ms = kernel_metrics(D, counts, per, hbm, bf16,
                                                      fused_route=layer.fused_route)
    achieved = kernels["expert_gemm1"]["gbs"]
    roofline = {"kernel": "expert_gemm1 (grouped GEMM 1 + clamped SwiGLU)", "bound": "hbm",
                "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": round(g1_bytes * GEMM1_DRAM_PER_ALGORITHMIC_BYTE),
                "traffic_source": "ncu dram read+write of a T=640/E=64 launch, scaled by bytes",
                "peak_source": peak_src, "bytes_per_launch": g1_bytes}
    ffn_launch = None
    if ffn_fused_supported(D.d, D.I):
        ffn_launch = {}
        for fused in (False, True):
            layer.fused_ffn = fused
            for _ in range(args.warmup):
                layer.experts()
            torch.cuda.synchronize()
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(args.steps):
                layer.experts()
            f1.record(stream)
            torch.cuda.synchronize()
            ffn_launch["one_launch_ms" if fused else "two_launches_ms"] = round(
                f0.elapsed_time(f1) / args.steps, 4)
        layer.fused_ffn = False
        assert _lib.moe_last_device_status() == _lib.MOE_OK
    # the same forward with the literal U(-0.1, 0.1) routing bias
    lw = W.scaled(wl, name=wl.name + "_bias0.1", bias_amp=0.1)
    lbias = W.make_inputs(lw, device=dev, with_weights=False)["bias"]
    for _ in range(args.warmup):
        layer.forward(inp["x"], lbias, inp["is_vision"], inp["logit_offset"])
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(args.steps):
        layer.forward(inp["x"], lbias, inp["is_vision"], inp["logit_offset"])
    l1.record(stream)
    torch.cuda.synchronize()
    lms = l0.elapsed_time(l1) / args.steps
    lc = layer.counts.cpu().numpy()
    literal = {"workload": f"{lw.name}: bias ~ U(-0.1, 0.1)",
               "value": round(replica_throughput(world, D.T, lms), 1), "unit": "tokens/s",
               "ms_per_step": round(lms, 4), "experts_with_tokens": int((lc > 0).sum()),
               "max_rows_per_expert": int(lc.max())}
    # forward passes over host batches: HostPipeline overlaps each batch's
    # copies with the neighbouring batches' compute
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty(D.T, D.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    pipe = HostPipeline(layer)
    route_args = (inp["bias"], inp["is_vision"], inp["logit_offset"])
    pipe.run([x_host] * args.warmup, [y_host[i % 2] for i in range(args.warmup)], *route_args)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run([x_host] * args.steps, [y_host[i % 2] for i in range(args.steps)], *route_args)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    out = {"workload": f"{wl.name}: forward, T={wl.T} d={wl.d} E={wl.E} routed top-{wl.k} + 1 "
                       f"shared, I={wl.I}, bias U(-0.01, 0.01)",
           "value": round(replica_throughput(world, D.T, ms_step), 1), "unit": "tokens/s",
           "ms_per_step": round(ms_step, 4), "roofline": roofline,
           "layer_roofline_ms": round(layer_roof_ms, 4),
           "layer_roofline_frac": round(layer_roof_ms / ms_step, 4), "kernels": kernels,
           "host_pipeline": {"value": round(replica_throughput(world, D.T, e2e_ms), 1),
                             "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                             "h2d_bytes_per_step": D.T * D.d * 2,
                             "d2h_bytes_per_step": D.T * D.d * 2},
           "literal_bias": literal, "expert_ffn_launches": ffn_launch,
           "routing": ("one kernel: gate projection + top-k + per-modality load (moe_gate_route)"
                       if layer.fused_route else "gate GEMM, then the routing kernel (moe_route)"),
           "expert_load": {"experts_with_tokens": int((counts > 0).sum()),
                           "min_rows": int(counts.min()), "max_rows": int(counts.max())}}
    del layer, pipe, x_host, y_host, inp
    torch.cuda.empty_cache()
    return out


def run_mx(args, weights, dev, world, hbm, bf16, names):
    """The MXFP8 forward (weights quantised once, token rows quantised in the
    dispatch, both expert matmuls on MXFP8 operands) on the named workloads,
    with the same per-call breakdown as the bf16 forward."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import Dims, MoELayer
    out = {}
    for name in names:
        wl = W.WORKLOADS[name]
        D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
        inp = layer_inputs(wl, dev, weights=weights)
        layer = MoELayer(D, weights, wl.rho, wl.clamp, mx=True)
        steps = args.steps if name == "full_fwd" else max(3, args.steps // 3)
        forward_breakdown(layer, inp, 1, args.warmup, world=world)
        counts = layer.counts.cpu().numpy()
        per, ms = forward_breakdown(layer, inp, steps, 1, world=world)
        assert _lib.moe_last_device_status() == _lib.MOE_OK
        kern, _, roof = kernel_metrics(D, counts, per, hbm, bf16,
                                       fused_route=layer.fused_route, mx=True)
        out[name] = {"workload": f"{name}: forward, MXFP8 expert matmuls, T={wl.T}",
                     "value": round(replica_throughput(world, D.T, ms), 1), "unit": "tokens/s",
                     "ms_per_step": round(ms, 4), "layer_roofline_ms": round(roof, 4),
                     "layer_roofline_frac": round(roof / ms, 4), "kernels": kern,
                     "steps": steps, "dtype": "mxfp8 operands (e4m3 + e8m0 per 32), fp32 accumulate"}
        del layer, inp
        torch.cuda.empty_cache()
    return out


def run_mx_only(args):
    """Only the MXFP8 forward of the workload (profiling captures)."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300.layer import Dims, MoELayer
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    hbm, bf16, _, _ = peaks()
    wl = workload(args)
    D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
    inp = layer_inputs(wl, dev)
    layer = MoELayer(D, {k: inp[k] for k in ("W_g", "W13", "W2")}, wl.rho, wl.clamp, mx=True)
    forward_breakdown(layer, inp, 1, args.warmup)
    counts = layer.counts.cpu().numpy()
    per, ms = forward_breakdown(layer, inp, args.steps, 1)
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    kern, _, roof = kernel_metrics(D, counts, per, hbm, bf16, fused_route=layer.fused_route,
                                   mx=True)
    return {"workload": f"{wl.name}: forward, MXFP8 expert matmuls", "ms_per_step": round(ms, 4),
            "value": round(D.T / ms * 1e3, 1), "unit": "tokens/s",
            "layer_roofline_frac": round(roof / ms, 4), "kernels": kern}


MX_STEP_CALLS = ["quantize_weights", "route", "dispatch", "expert_gemm1", "expert_gemm2",
                 "combine"]
MX_MATMUL_STAGES = {"expert_gemm1", "expert_gemm2", "bwd_recompute_gemm1", "bwd_dgrad2",
                    "bwd_dgrad1", "bwd_wgrad2", "bwd_wgrad1"}


def mx_step_work(D, counts):
    """Algorithmic FLOPs and minimum HBM bytes of each call of the MXFP8
    training step (codes one byte an element, scales one byte per 32)."""
    used = int((counts > 0).sum()) + 1
    R, S, T, d, I, E, G = D.R, D.S, D.T, D.d, D.I, D.E, D.E + 1
    nw = 3 * G * d * I                               # weight elements
    sc = lambda n: n // 32                           # scale bytes of n elements
    fwd = {
        "quantize_weights": (0, nw * 2 + 2 * (nw + sc(nw))),   # one read, both copies
        "route": (2 * T * d * E, T * d * 2 + E * d * 2 + T * E * 4 + T * D.k * 12),
        "dispatch": (0, T * d * 2 + R * d + sc(R * d) + S * 4 * 6),
        "expert_gemm1": (4 * R * d * I, used * 2 * I * d + R * d + sc(R * d) + R * I + sc(R * I)),
        "expert_gemm2": (2 * R * I * d, used * d * I + R * I + sc(R * I) + R * d * 2),
        "combine": (0, R * d * 2 + T * d * 2 + S * 4),
    }
    bwd = {
        "recompute_gather": (0, T * d * 2 + R * d * 2),
        "recompute_gemm1": (4 * R * d * I, used * 2 * I * d + R * d + R * 2 * I * 4 + R * I),
        "gather_dY": (0, T * d * 2 + R * d + sc(R * d)),
        "dgrad2": (2 * R * d * I, used * d * I + R * d + R * 2 * I * 4 + R * I
                   + R * 2 * I * 2 + R * 2 * I + R * I * 2),
        # the operands quantised along the rows (read bf16, write codes, read
        # the codes back in the matmul), then fp32 dW2
        "wgrad2": (2 * R * d * I, T * d * 2 + R * I * 2 + 2 * (d + I) * R + G * d * I * 4),
        "dgrad1": (4 * R * I * d, used * 2 * I * d + R * 2 * I + R * d * 2),
        "wgrad1": (4 * R * I * d, R * 2 * I * 2 + R * d * 2 + 2 * (2 * I + d) * R
                   + G * 2 * I * d * 4),
        "router_bwd": (0, S * 4 * 6 + T * E * 4),
        "dX": (2 * S * d, R * d * 2 + T * d * 2 + S * 8),
        "dW_g": (2 * S * d, S * d * 2 + E * d * 4),
    }
    return fwd, bwd


def run_mx_fwd_bwd(args, weights, dev, world, hbm, bf16_sus, wl=None):
    """One MXFP8 training step of the workload (the headline's by default):
    the expert weights quantised from bf16 (both orientations, as after an
    optimizer update), the forward with MX expert matmuls and the MX backward
    (dgrad and weight-gradient matmuls on MX operands), CUDA events around
    each call and backward stage."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import Dims, MoELayer
    wl = wl or W.WORKLOADS[HEADLINE]
    D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
    inp = layer_inputs(wl, dev, weights=weights)
    if weights is None:
        weights = {k: inp[k] for k in ("W_g", "W13", "W2")}
    layer = MoELayer(D, weights, wl.rho, wl.clamp, backward=True, recompute=wl.recompute,
                     mx=True)
    stream = torch.cuda.current_stream()
    nb = _lib.MOE_BWD_STAGES
    off = inp["logit_offset"]

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    def step(fev=None, bev=None):
        def mark(i):
            if fev is not None:
                fev[i].record(stream)
        mark(0)
        layer.quantize_weights()
        mark(1)
        layer.route(inp["x"], inp["bias"], inp["is_vision"], off)
        mark(2)
        layer.dispatch(inp["x"])
        mark(3)
        layer.expert_gemm1()
        mark(4)
        layer.expert_gemm2()
        mark(5)
        layer.combine()
        mark(6)
        layer.backward(inp["dY"], stage_events=bev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    counts = layer.counts.cpu().numpy()
    K = max(3, args.steps // 2)
    fevs = [events(len(MX_STEP_CALLS) + 1) for _ in range(K)]
    bevs = [events(nb + 1) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(fevs[i], bevs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    ms = dist_max(t0.elapsed_time(t1) / K, world)
    fwd_ms = {n: sum(fevs[i][j].elapsed_time(fevs[i][j + 1]) for i in range(K)) / K
              for j, n in enumerate(MX_STEP_CALLS)}
    bwd_ms = {n: sum(bevs[i][j].elapsed_time(bevs[i][j + 1]) for i in range(K)) / K
              for j, n in enumerate(_lib.MOE_BWD_STAGE_NAMES)}
    fwd_work, bwd_work = mx_step_work(D, counts)
    kernels = {}
    for n in MX_STEP_CALLS:
        peak = 2 * bf16_sus if n in MX_MATMUL_STAGES else bf16_sus
        kernels[n] = stage_metrics(fwd_ms[n], *fwd_work[n], hbm, peak)
    for n in _lib.MOE_BWD_STAGE_NAMES:
        if bwd_ms[n] > 0:
            key = "bwd_" + n
            peak = 2 * bf16_sus if key in MX_MATMUL_STAGES else bf16_sus
            kernels[key] = stage_metrics(bwd_ms[n], *bwd_work[n], hbm, peak)
    out = {"workload": f"{wl.name}: MXFP8 training step (weights quantised, forward, "
                       f"backward), T={wl.T} d={wl.d} E={wl.E} top-{wl.k} + shared, I={wl.I}"
                       + (", recompute" if wl.recompute else ""),
           "value": round(replica_throughput(world, D.T, ms), 1), "unit": "tokens/s",
           "ms_per_step": round(ms, 4), "steps": K,
           "dtype": "mxfp8 operands (e4m3 + e8m0 per 32) in every matmul of the step, "
                    "fp32 accumulate, fp32 weight gradients",
           "peak_note": "MX matmul stages against 2x the measured sustained bf16 peak",
           "kernels": kernels}
    del layer, inp
    torch.cuda.empty_cache()
    return out


def run_mx_fwd_bwd_only(args):
    """Only the MXFP8 training step of the workload (profiling captures)."""
    from moe_expert_layer_04_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    hbm, _, bf16_sus, _ = peaks()
    wl = workload(args)
    return run_mx_fwd_bwd(args, None, dev, 1, hbm, bf16_sus, wl=wl)


def run_extra_workloads(args, weights, dev, world, hbm, bf16):
    """Per-call numbers of the skewed multimodal forward (top-k and hash
    routing), one of the sizes where the HBM targets of the routing /
    dispatch / combine steps apply."""
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH, Dims, MoELayer
    steps = max(3, args.steps // 3)
    out = {}
    for name, modes in (("skewed_mm_fwd", (0, MOE_ROUTE_HASH)),):
        wl = W.WORKLOADS[name]
        D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
        inp = layer_inputs(wl, dev, weights=weights)
        layer = MoELayer(D, weights, wl.rho, wl.clamp)
        for mode in modes:
            per, ms = forward_breakdown(layer, inp, steps, args.warmup, mode=mode, world=world)
            counts = layer.counts.cpu().numpy()
            kern, _, roof = kernel_metrics(D, counts, per, hbm, bf16,
                                           fused_route=layer.fused_route)
            key = name + ("_hash" if mode == MOE_ROUTE_HASH else "")
            load = {"experts_with_tokens": int((counts > 0).sum()), "max_rows": int(counts.max())}
            if layer.modality_counts is not None:
                mc = layer.modality_counts.cpu().numpy()
                # text and vision slots per expert, from the routing kernel's counters
                load["by_modality"] = {m: {"slots": int(mc[i].sum()), "max_rows": int(mc[i].max()),
                                           "experts_with_tokens": int((mc[i] > 0).sum())}
                                       for i, m in enumerate(("text", "vision"))}
            out[key] = {"workload": f"{name}: forward, T={wl.T}" +
                                    (", hash router" if mode == MOE_ROUTE_HASH else ", top-k router"),
                        "value": round(replica_throughput(world, D.T, ms), 1),
                        "unit": "tokens/s",
                        "ms_per_step": round(ms, 4), "layer_roofline_frac": round(roof / ms, 4),
                        "kernels": kern, "steps": steps, "expert_load": load}
        del layer
        torch.cuda.empty_cache()
        if wl.backward and not args.no_bwd:
            out[name + "_fwd_bwd"] = run_fwd_bwd(args, weights, dev, world, wl_name=name,
                                                 inputs=inp)
        del inp
        torch.cuda.empty_cache()
    return out


def run_fwd_bwd(args, weights, dev, world, wl_name="fwd_bwd", inputs=None, wl=None):
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import Dims, MoELayer
    if wl is None:
        wl = W.WORKLOADS[wl_name]
        over = {k: v for k, v in (("T", args.tokens), ("E", args.experts)) if v}
        if over:
            wl = W.scaled(wl, name=wl.name + "-" + "-".join(f"{k}{v}" for k, v in over.items()),
                          **over)
    D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
    inp = inputs if inputs is not None else layer_inputs(wl, dev, weights=weights)
    layer = MoELayer(D, weights, wl.rho, wl.clamp, backward=True, recompute=wl.recompute)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
        if ev is not None:
            ev.record(stream)
        layer.backward(inp["dY"])

    steps = max(3, args.steps // 2)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    dist_barrier(world)
    torch.cuda.synchronize()
    starts[0].record(stream)
    for i in range(steps):
        step(mids[i])
        starts[i + 1].record(stream)
    torch.cuda.synchronize()
    ms = starts[0].elapsed_time(starts[-1]) / steps
    bwd_ms = sum(mids[i].elapsed_time(starts[i + 1]) for i in range(steps)) / steps
    ms = dist_max(ms, world)
    out = {"workload": f"{wl.name}: forward+backward, T={wl.T} d={wl.d} E={wl.E} top-{wl.k} "
                       f"+ shared, I={wl.I}, fp32 weight grads"
                       + (", recompute" if wl.recompute else ""),
           "value": round(replica_throughput(world, D.T, ms), 1), "unit": "tokens/s",
           "ms_per_step": round(ms, 4), "bwd_ms": round(bwd_ms, 4), "steps": steps,
           "gpu_launches": (fwd_launches(layer.fused_route) + BWD_LAUNCHES
                            + (BWD_RECOMPUTE_EXTRA if wl.recompute else 0)) * steps}
    del layer, inp
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------ the headline step

HEADLINE = "long_slice_fwd_bwd"
FWD_CALLS = ["route", "permute", "expert_gemm1", "expert_gemm2", "combine"]


def bwd_stage_work(D, counts):
    """Algorithmic FLOPs and minimum HBM bytes of each moe_backward stage:
    weights of every expert with rows read once, fp32 weight gradients
    written once, each permuted activation read or written once."""
    from moe_expert_layer_04_gb300 import _lib
    used = int((counts > 0).sum()) + 1
    R, S, T, d, I, E = D.R, D.S, D.T, D.d, D.I, D.E
    w13, w2 = used * 2 * I * d * 2, used * d * I * 2
    work = {
        "recompute_gather": (0, T * d * 2 + R * d * 2),
        "recompute_gemm1": (4 * R * d * I, w13 + R * d * 2 + R * 2 * I * 4),
        "gather_dY": (0, T * d * 2 + R * d * 2),
        "dgrad2": (2 * R * d * I, w2 + R * d * 2 + R * 2 * I * 4 + R * 2 * I * 2 + R * I * 2),
        "wgrad2": (2 * R * d * I, (E + 1) * d * I * 4 + R * d * 2 + R * I * 2),
        "dgrad1": (4 * R * I * d, w13 + R * 2 * I * 2 + R * d * 2),
        "wgrad1": (4 * R * I * d, (E + 1) * 2 * I * d * 4 + R * 2 * I * 2 + R * d * 2),
        "router_bwd": (0, S * 4 * 6 + T * E * 4),
        "dX": (2 * S * d, R * d * 2 + T * d * 2 + S * 8),
        "dW_g": (2 * S * d, S * d * 2 + E * d * 4),
    }
    assert list(work) == _lib.MOE_BWD_STAGE_NAMES
    return work


def stage_metrics(ms, flops, nbytes, hbm, tflops_peak):
    sec = ms / 1e3
    m = {"ms": round(ms, 4), "gbs": round(nbytes / sec / 1e9, 1),
         "hbm_frac": round(nbytes / sec / 1e9 / hbm, 4)}
    if flops:
        m["tflops"] = round(flops / sec / 1e12, 1)
        m["tensor_frac"] = round(flops / sec / 1e12 / tflops_peak, 4)
    return m


def oracle_fwd_bwd_sample(host, wl, n_tok, n_rows, rng):
    """The oracle on a bounded sample of a forward + backward step: the
    forward and the token-local backward (dX, logit and routing-weight
    gradients) of n_tok seeded tokens, and the weight gradients of the shared
    expert over n_rows seeded token rows (one output of each weight gradient,
    as a full step writes it once per expert).  A token's share of a step is
    its forward and local backward plus k + 1 weight-gradient rows (its k
    routed experts and the shared one).  Returns (seconds of CPU work,
    seconds per token)."""
    import oracle
    tok = np.sort(rng.choice(wl.T, size=min(n_tok, wl.T), replace=False))
    rows = np.sort(rng.choice(wl.T, size=min(n_rows, wl.T), replace=False))
    kw = dict(is_vision=host["is_vision"], offset=host["logit_offset"])
    t0 = time.perf_counter()
    oracle.layer_forward(host["x"], host["W_g"], host["W13"], host["W2"], host["bias"], wl.k,
                         wl.rho, wl.clamp, tok=tok, **kw)
    oracle.layer_backward(host["x"], host["W_g"], host["W13"], host["W2"], host["dY"],
                          host["bias"], wl.k, wl.rho, wl.clamp, tok=tok, **kw)
    t1 = time.perf_counter()
    oracle.expert_wgrad(host["x"], host["W13"], host["W2"], host["dY"], wl.E, rows,
                        np.ones(len(rows)), wl.clamp)
    t2 = time.perf_counter()
    per_tok = (t1 - t0) / len(tok) + (wl.k + 1) * (t2 - t1) / len(rows)
    return t2 - t0, per_tok


def cpu_baseline_fwd_bwd(inp, wl, n_tok, n_rows):
    import oracle
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    oracle.build()
    sec, per_tok = oracle_fwd_bwd_sample(host, wl, n_tok, n_rows, np.random.default_rng(0))
    return {"value": round(1.0 / per_tok, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"forward + token-local backward of {n_tok} seeded tokens and the weight "
                      f"gradients of the shared expert over {n_rows} seeded token rows of the "
                      f"{wl.name} workload; a token costs its forward and local backward plus "
                      f"k + 1 = {wl.k + 1} weight-gradient rows ({sec:.1f} s of CPU work, "
                      f"OpenMP over tokens / output entries)"}


def run_headline(args, weights, dev, world, hbm, bf16_sus):
    """The headline: forward + backward of the 64K-token slice, with CUDA
    events around each forward call and each backward stage."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import Dims, MoELayer
    wl = W.WORKLOADS[HEADLINE]
    over = {k: v for k, v in (("T", args.tokens), ("E", args.experts)) if v}
    if over:
        wl = W.scaled(wl, name=wl.name + "-" + "-".join(f"{k}{v}" for k, v in over.items()), **over)
    D = Dims(wl.T, wl.d, wl.E, wl.k, wl.I)
    inp = layer_inputs(wl, dev, weights=weights)
    layer = MoELayer(D, weights, wl.rho, wl.clamp, backward=True, recompute=wl.recompute)
    stream = torch.cuda.current_stream()
    nb = _lib.MOE_BWD_STAGES
    off = inp["logit_offset"]

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)      # creates the CUDA event behind each
        return evs

    def step(fev=None, bev=None):
        def mark(i):
            if fev is not None:
                fev[i].record(stream)
        mark(0)
        layer.route(inp["x"], inp["bias"], inp["is_vision"], off)
        mark(1)
        layer.dispatch(inp["x"])
        mark(2)
        layer.expert_gemm1()
        mark(3)
        layer.expert_gemm2()
        mark(4)
        layer.combine()
        mark(5)
        layer.backward(inp["dY"], stage_events=bev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    counts = layer.counts.cpu().numpy()
    K = args.steps
    fevs = [events(6) for _ in range(K)]
    bevs = [events(nb + 1) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(fevs[i], bevs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    ms_step = dist_max(t0.elapsed_time(t1) / K, world)
    fwd_ms = {n: sum(fevs[i][j].elapsed_time(fevs[i][j + 1]) for i in range(K)) / K
              for j, n in enumerate(FWD_CALLS)}
    bwd_ms = {n: sum(bevs[i][j].elapsed_time(bevs[i][j + 1]) for i in range(K)) / K
              for j, n in enumerate(_lib.MOE_BWD_STAGE_NAMES)}

    # per call / stage: algorithmic work against the sustained peaks (the
    # kernels run inside a step of tens of milliseconds)
    g1b, g2b = fwd_algorithmic_bytes(D, counts)
    fwd_work = {"route": (2 * D.T * D.d * D.E, D.T * D.d * 2 + D.E * D.d * 2 + D.T * D.E * 4
                          + D.T * D.k * 12),
                "permute": (0, D.T * D.d * 2 + D.R * D.d * 2 + D.S * 4 * 6),
                "expert_gemm1": (4 * D.R * D.d * D.I, g1b),
                "expert_gemm2": (2 * D.R * D.I * D.d, g2b),
                "combine": (0, D.R * D.d * 2 + D.T * D.d * 2 + D.S * 4)}
    bwd_work = bwd_stage_work(D, counts)
    kernels = {n: stage_metrics(fwd_ms[n], *fwd_work[n], hbm, bf16_sus) for n in FWD_CALLS}
    kernels.update({"bwd_" + n: stage_metrics(bwd_ms[n], *bwd_work[n], hbm, bf16_sus)
                    for n in _lib.MOE_BWD_STAGE_NAMES if bwd_ms[n] > 0})

    # the dominant kernel: the grouped-GEMM kernel (template instance) with the
    # largest share of the step
    groups = {
        "expert GEMM 1 (moe_gemm_kernel<GM_FFN1>: forward and the backward's recompute)":
            (("fwd", "expert_gemm1"), ("bwd", "recompute_gemm1")),
        "weight gradients (moe_gemm_kernel<GM_WGRAD>: dW2 and dW13)":
            (("bwd", "wgrad2"), ("bwd", "wgrad1")),
        "dgrad 1 (moe_gemm_kernel<GM_DGRAD1>)": (("bwd", "dgrad1"),),
        "dgrad 2 + SwiGLU backward (moe_gemm_kernel<GM_DGRAD2>)": (("bwd", "dgrad2"),),
        "expert GEMM 2 (moe_gemm_kernel<GM_FFN2>)": (("fwd", "expert_gemm2"),),
    }
    def tot(parts, what):
        out = 0.0
        for side, n in parts:
            if side == "fwd":
                out += fwd_ms[n] if what == "ms" else fwd_work[n][0]
            else:
                out += bwd_ms[n] if what == "ms" else bwd_work[n][0]
        return out
    name = max(groups, key=lambda g: tot(groups[g], "ms"))
    g_ms, g_fl, n_launch = tot(groups[name], "ms"), tot(groups[name], "flops"), len(groups[name])
    achieved = g_fl / (g_ms / 1e3) / 1e12
    traffic = None
    if wl.name == HEADLINE and not args.tokens and not args.experts:
        traffic = next((round(v) for k, v in LONG_SLICE_DRAM_BYTES_PER_LAUNCH.items()
                        if name.startswith(k)), None)
    roofline = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": bf16_sus, "unit": "TFLOP/s", "frac": round(achieved / bf16_sus, 4),
                "traffic": traffic,
                "traffic_source": "ncu dram read+write per launch at this workload "
                                  "(profiles/dram_traffic_long_slice_fwd_bwd.md)",
                "launches_per_step": n_launch,
                "flops_per_launch": int(g_fl / n_launch),
                "ms_per_launch": round(g_ms / n_launch, 4),
                "peak_source": "measured sustained bf16 (cuBLAS loop under the power cap)"}
    alg_flops = (sum(fwd_work[n][0] for n in FWD_CALLS) +
                 sum(f for n, (f, _) in bwd_work.items() if n != "recompute_gemm1"))
    layer_roof_ms = alg_flops / (bf16_sus * 1e12) * 1e3
    out = dict(wl=wl, D=D, inp=inp, layer=layer, ms_step=ms_step, kernels=kernels,
               roofline=roofline, counts=counts, layer_roof_ms=layer_roof_ms,
               alg_flops=alg_flops,
               launches=fwd_launches(layer.fused_route) + BWD_LAUNCHES +
               (BWD_RECOMPUTE_EXTRA if wl.recompute else 0))
    return out


def run_headline_e2e(args, h, world):
    """The headline step end to end through the C ABI with host buffers: x
    and dY copied in from pinned host memory and y and dX copied back every
    step.  moe_layer_steps_host pipelines the steps (the next step's uploads
    and the last step's downloads overlap the compute; two sets of host
    buffers in turn); moe_layer_step_host, one step per call, is timed beside
    it."""
    layer, inp, D = h["layer"], h["inp"], h["D"]
    stream = torch.cuda.current_stream()
    x_h = [inp["x"].cpu().pin_memory() for _ in range(2)]
    dY_h = [inp["dY"].cpu().pin_memory() for _ in range(2)]
    y_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(2)]
    dX_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(2)]
    ci, co = torch.cuda.Stream(), torch.cuda.Stream()
    route = dict(bias=inp["bias"], is_vision=inp["is_vision"], logit_offset=inp["logit_offset"])

    def steps(n):
        pick = lambda b: [b[i % 2] for i in range(n)]
        layer.steps_host(pick(x_h), pick(y_h), pick(dY_h), pick(dX_h), copy_in_stream=ci,
                         copy_out_stream=co, **route)

    def timed(fn):
        torch.cuda.synchronize()
        dist_barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return dist_max(e0.elapsed_time(e1) / args.steps, world)

    steps(args.warmup)
    ms = timed(lambda: steps(args.steps))
    cs = torch.cuda.Stream()

    def one_by_one():
        for i in range(args.steps):
            layer.step_host(x_h[i % 2], y_h[i % 2], dY_h[i % 2], dX_h[i % 2], copy_stream=cs,
                            **route)
    one_by_one()
    ms1 = timed(one_by_one)
    nb = D.T * D.d * 2
    return {"value": round(replica_throughput(world, D.T, ms), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": 2 * nb, "d2h_bytes_per_step": 2 * nb,
            "ms_per_step": round(ms, 4),
            "path": "moe_layer_steps_host (C ABI; host x and dY in, host y and dX out every "
                    "step; the next step's uploads and the last step's downloads overlap "
                    "the compute)",
            "one_step_per_call_ms": round(ms1, 4)}


# --------------------------------------------- forward + backward alone

def run_fwd_bwd_only(args):
    """Forward + backward of the named workload alone (its own weights at its
    own sizes), e.g. to capture a launch list of the 64K-token slice."""
    from moe_expert_layer_04_gb300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    wl = workload(args)
    inp = layer_inputs(wl, dev)
    weights = {k: inp[k] for k in ("W_g", "W13", "W2")}
    args.tokens = args.experts = 0          # already applied by workload()
    out = run_fwd_bwd(args, weights, dev, 1, wl_name=args.workload, inputs=inp, wl=wl)
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return out


# ------------------------------------------------------ routing alone

def run_route_only(args):
    """Times the routing step alone (gate projection + routing) on the
    workload's routing inputs: the one-kernel path (moe_gate_route, with the
    per-modality counters) and the two-kernel path (moe_route), CUDA events
    around each call, L2 flushed before each.  Used to profile the routing
    kernels without the expert weights on the device."""
    from moe_expert_layer_04_gb300 import _lib
    from moe_expert_layer_04_gb300 import workloads as W
    from moe_expert_layer_04_gb300.layer import gate_route_supported
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workload(args)
    inp = W.make_inputs(wl, device=dev, with_weights=False)
    Wg = W.normal_bf16((wl.E, wl.d), 0.02, wl.seed, "W_g", dev)
    T, E, k = wl.T, wl.E, wl.k
    z = torch.empty(T, E, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, k, device=dev)
    ssel = torch.empty(T, k, device=dev)
    cnt = torch.empty(2, E, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    args_r = (inp["x"], Wg, inp["logit_offset"], inp["bias"], inp["is_vision"], None, None, T,
              wl.d, E, k, wl.rho, 0, z, ids, wts, ssel)
    paths = [("two_kernels", lambda: _lib.moe_route(*args_r))]
    if gate_route_supported(wl.d, E, k):
        paths.insert(0, ("fused", lambda: _lib.moe_gate_route(*args_r, cnt)))
    out = {}
    for name, call in paths:
        for _ in range(args.warmup):
            call()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        assert _lib.moe_last_device_status() == _lib.MOE_OK
        out[name] = {"ms": round(statistics.median(ts), 4),
                     "tflops": round(2 * T * wl.d * E / (statistics.median(ts) / 1e3) / 1e12, 1)}
    return {"metric": "routing step ms (gate projection + top-k routing)",
            "config": {"workload": f"{wl.name}: T={T} d={wl.d} E={E} top-{k}"},
            "steps": args.steps, "warmup": args.warmup, "l2": "flushed before each call",
            **out}


# -------------------------------------------------------------- oracle

def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample of the
    headline forward + backward (oracle_fwd_bwd_sample), its tokens/s the
    sample's tokens over the CPU time they cost."""
    import oracle
    from moe_expert_layer_04_gb300 import workloads as W
    if rank != 0:
        return None
    wl = W.WORKLOADS[HEADLINE]
    over = {k: v for k, v in (("T", args.tokens), ("E", args.experts)) if v}
    if over:
        wl = W.scaled(wl, name=wl.name + "-" + "-".join(f"{k}{v}" for k, v in over.items()), **over)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = layer_inputs(wl, dev)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    del inp
    if dev == "cuda":
        torch.cuda.empty_cache()
    oracle.build()
    rng = np.random.default_rng(1)
    n_tok, n_rows = args.ref_tokens, args.ref_rows
    for _ in range(args.warmup):
        oracle_fwd_bwd_sample(host, wl, n_tok, n_rows, rng)
    secs, per_tok = [], []
    for _ in range(args.steps):
        sec, pt = oracle_fwd_bwd_sample(host, wl, n_tok, n_rows, rng)
        secs.append(sec)
        per_tok.append(pt)
    value = round(1.0 / statistics.mean(per_tok), 3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(secs) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_string(wl), "global_batch": wl.T * world,
                   "seq_len": wl.T, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: forward + token-local backward of {n_tok} random "
                                   f"tokens and the shared expert's weight gradients over "
                                   f"{n_rows} random token rows; a token costs its forward and "
                                   f"local backward plus k + 1 weight-gradient rows"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    help="workload of the profiling modes (--route-only, --fwd-bwd-only, "
                         "--mx-only)")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the skewed and 64K-token workloads")
    ap.add_argument("--cpu-tokens", type=int, default=64,
                    help="oracle baseline: tokens of the forward + local backward sample")
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="oracle baseline: shared-expert rows of the weight-gradient sample")
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling)")
    ap.add_argument("--route-only", action="store_true",
                    help="time only the routing step of the workload (profiling)")
    ap.add_argument("--fwd-bwd-only", action="store_true",
                    help="time only forward + backward of the workload (profiling)")
    ap.add_argument("--no-mx", action="store_true", help="skip the MXFP8 forward")
    ap.add_argument("--mx-only", action="store_true",
                    help="time only the MXFP8 forward of the workload (profiling)")
    ap.add_argument("--mx-fwd-bwd-only", action="store_true",
                    help="time only the MXFP8 training step of the workload (profiling)")
    ap.add_argument("--pairs", type=int, default=None,
                    help="MOE_PAIR_* mask of the matmuls that may run as 2-SM pairs "
                         "(default: the library's)")
    args = ap.parse_args()
    if args.pairs is not None:
        from moe_expert_layer_04_gb300 import _lib
        _lib.moe_set_gemm_pairs(args.pairs)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.route_only:
        print(json.dumps(run_route_only(args)), flush=True)
        return
    if args.fwd_bwd_only:
        print(json.dumps(run_fwd_bwd_only(args)), flush=True)
        return
    if args.mx_only:
        print(json.dumps(run_mx_only(args)), flush=True)
        return
    if args.mx_fwd_bwd_only:
        print(json.dumps(run_mx_fwd_bwd_only(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
