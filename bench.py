#!/usr/bin/env python3
"""Benchmark: conv2d TFLOP/s per op (forward / backward-data / backward-filter) on GB300.

One step = the whole hot path once: forward, backward-data and backward-filter of the
workload (default: the largest of the five by FLOP, the bf16 deconvolution layer: deconv
input [32,512,16,16] -> output [32,256,32,32], weight [512,256,4,4], stride 2, pad 1) on
seeded synthetic inputs already resident in HBM.  Every workload's three ops are also
timed alone (the per_config block).
Each op is timed with CUDA events on the launching stream; L2 is flushed (a write of
twice the L2 size) before every op, outside the events.  FLOP per op = 2*N*K*P*Q*C*R*S.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle on a bounded
sample of the same workload instead (the slow, plainly correct reference arm).
Multi-GPU (torchrun, one rank per GPU): the path is run as independent replicas, one per
rank, no collective on the data path; value = all ranks' FLOP / max rank time.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv2d TFLOP/s per op (fwd/dgrad/wgrad) and % of GB300 tensor-core peak"
OPS = ("fwd", "bwd_data", "bwd_filter")
# The headline workload: the largest of the five by FLOP per op (the bf16 deconvolution layer,
# 3.44e10); every workload is timed in the line's per_config block.
DEFAULT_WORKLOAD = "deconv"
# Fallback peaks (used only if MEASURED_PEAKS.json is absent): one earlier GB300 measurement.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--config-reps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--profile", choices=OPS, default=None,
                    help="run only this op of the workload (warmup + steps calls) for a profiler; prints its mean ms")
    ap.add_argument("--groups", type=int, default=1,
                    help="with --profile: the workload's layer with this many groups (filter K x C/groups)")
    return ap.parse_args()


def run_profile(args):
    """One op of one workload, `warmup` + `steps` calls back to back (L2 flushed before each), for
    capturing its kernels under a profiler; prints the mean device time of the last `steps` calls."""
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    from convolution_nchw_conv2d_gb300 import workloads as W
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8, device=dev)
    c = _device_case(W.WORKLOADS[args.workload], dev)
    call = lambda: _op_call(c, args.profile, stream)
    if args.groups > 1:  # the same layer grouped: filter K x C/groups, each op's grouped call
        pb, g = c["pb"], args.groups
        pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
        dt = 0 if pb.dtype == "f32" else 1
        wg = c["w"][:, : pb.C // g].contiguous()
        dwg = torch.empty_like(wg)
        wsz = max(cg.conv2d_workspace_size(op, pb.dims(), dt, (1, 1), g) for op in range(3))
        wsg = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
        calls = {"fwd": lambda: cg.conv2d_fwd(c["x"], wg, pad, st, out=c["y"], workspace=wsg, stream=stream, groups=g),
                 "bwd_data": lambda: cg.conv2d_bwd_data(c["dy"], wg, (pb.H, pb.W), pad, st, out=c["dx"], workspace=wsg,
                                                        stream=stream, groups=g),
                 "bwd_filter": lambda: cg.conv2d_bwd_filter(c["x"], c["dy"], (pb.R, pb.S), pad, st, out=dwg,
                                                            workspace=wsg, stream=stream, groups=g)}
        call = calls[args.profile]
    ms = _time_call(call, flush, stream, max(1, args.steps), args.warmup)
    cg.conv2d_device_status(stream)
    print(json.dumps({"profile": args.profile, "workload": args.workload, "groups": args.groups, "ms": round(ms, 5)}),
          flush=True)
    return 0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf = d.get("bf16_tflops")
            if hbm and bf:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf),
                        "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", bf)),
                        "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK, source="fallback")


def src_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "convolution_nchw_conv2d_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, op):
    """DRAM bytes per launch from the committed ncu summary, if taken on this source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{workload}/{op}")
        if e and e.get("source_sha") == src_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        all_sm = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk = float(parts[2])
                cmax = float(parts[3])
            except ValueError:
                continue
            all_sm.append((ts, clk, cmax, parts[6:10]))
        inside = [s for s in all_sm if t0 - 0.15 <= s[0] <= t1 + 0.15] or all_sm
        for ts, clk, cmax, flags in inside:
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, flags):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def slowest_rank_ms(ms, world, device):
    """Replicas only: every rank runs the whole step on its own GPU; the job's step time is the
    slowest rank's (MAX over ranks through the process group; no data-path collective)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_op, n_ops, world, step_ms):
    """Whole-job throughput: all ranks' FLOP over the slowest rank's step time (weak scaling)."""
    return world * n_ops * flop_per_op / (step_ms * 1e-3) / 1e12


def _device_case(wl, dev):
    """Seeded inputs of a workload on the device, its outputs and one workspace for all three ops."""
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    from convolution_nchw_conv2d_gb300 import workloads as W
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    c = {"pb": pb, "host": (x, w, dy), "x": x.to(dev), "w": w.to(dev), "dy": dy.to(dev),
         "y": torch.empty(pb.y_shape, dtype=x.dtype, device=dev),
         "dx": torch.empty(pb.x_shape, dtype=x.dtype, device=dev),
         "dw": torch.empty(pb.w_shape, dtype=x.dtype, device=dev)}
    dt = 0 if pb.dtype == "f32" else 1
    wsz = max(cg.conv2d_workspace_size(op, pb.dims(), dt) for op in range(3))
    c["ws"] = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)
    return c


def _op_call(c, op, stream):
    import convolution_nchw_conv2d_gb300 as cg
    pb = c["pb"]
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    if op == "fwd":
        cg.conv2d_fwd(c["x"], c["w"], pad, st, out=c["y"], workspace=c["ws"], stream=stream)
    elif op == "bwd_data":
        cg.conv2d_bwd_data(c["dy"], c["w"], (pb.H, pb.W), pad, st, out=c["dx"], workspace=c["ws"], stream=stream)
    else:
        cg.conv2d_bwd_filter(c["x"], c["dy"], (pb.R, pb.S), pad, st, out=c["dw"], workspace=c["ws"], stream=stream)


def _time_call(fn, flush, stream, reps, warmup):
    """Mean device time (ms) of fn over `reps` calls, CUDA events on `stream` around each call;
    L2 flushed (a write of twice its size) before every call, outside the events."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    pairs = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs) / len(pairs)


def _roofline_of(pb, op_ms, peaks):
    """Per-op throughput and fractions of the tensor and HBM peaks; the dominant (slowest) op
    against whichever roof bounds it (tensor when its arithmetic intensity is past the ridge)."""
    tc_peak = peaks["bf16_tflops"] * (NOMINAL_TF32_OVER_BF16 if pb.dtype == "f32" else 1.0)
    flop = pb.flops()
    per_op = {}
    for op in OPS:
        tf = flop / (op_ms[op] * 1e-3) / 1e12
        gbs = pb.alg_bytes(op) / (op_ms[op] * 1e-3) / 1e9
        per_op[op] = {"ms": round(op_ms[op], 5), "tflops": round(tf, 2),
                      "frac_tc_peak": round(tf / tc_peak, 4), "alg_gbs": round(gbs, 1),
                      "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)}
    dom = max(OPS, key=lambda o: op_ms[o])
    ai = flop / pb.alg_bytes(dom)
    if ai * peaks["hbm_gbs"] * 1e9 < tc_peak * 1e12:
        roof = {"bound": "hbm", "achieved": per_op[dom]["alg_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": per_op[dom]["tflops"], "peak": round(tc_peak, 1), "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["kernel"] = dom
    return per_op, roof


def _fused_backward(c, flush, stream, reps, warmup, op_ms):
    """Both gradients through the one-call backward (dy read once where the plans share it) beside
    the two separate backward calls on the same workload."""
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    pb = c["pb"]
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    dt = 0 if pb.dtype == "f32" else 1
    wsz = cg.conv2d_workspace_size(cg.OP_BWD, pb.dims(), dt)
    ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device=c["x"].device)
    ms = _time_call(lambda: cg.conv2d_bwd(c["x"], c["w"], c["dy"], pad, st, dx=c["dx"], dw=c["dw"], workspace=ws,
                                          stream=stream), flush, stream, reps, warmup)
    sep = op_ms["bwd_data"] + op_ms["bwd_filter"]
    return {"bwd_ms": round(ms, 5), "bwd_data_plus_bwd_filter_ms": round(sep, 5),
            "tflops": round(2 * pb.flops() / (ms * 1e-3) / 1e12, 2), "saved_ms": round(sep - ms, 5),
            "note": "conv2d_bwd (dx and dw in one call) against the two separate calls, same inputs"}


def _extras_resnet(c, flush, stream, reps, warmup, op_ms):
    """Timings of the extended entry points on the ResNet 3x3 layer: the fused epilogues (bias +
    add-to on the forward op, both bias gradients on backward-filter), dilation 2, groups 2."""
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    pb = c["pb"]
    dev = c["x"].device
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    dt = 0 if pb.dtype == "f32" else 1
    x, w, dy, y, dx, dw, ws = c["x"], c["w"], c["dy"], c["y"], c["dx"], c["dw"], c["ws"]
    bias_k = torch.randn(pb.K, generator=torch.Generator().manual_seed(5)).to(x.dtype).to(dev)
    dbk = torch.empty(pb.K, dtype=x.dtype, device=dev)
    dbc = torch.empty(pb.C, dtype=x.dtype, device=dev)
    wsz_f = cg.conv2d_workspace_size(2, pb.dims(), dt)
    ws_f = torch.empty(max(wsz_f, 16), dtype=torch.uint8, device=dev) if wsz_f > ws.numel() else ws
    ex_ms = {
        "fwd_bias_addto": _time_call(lambda: cg.conv2d_fwd(x, w, pad, st, out=y, workspace=ws, stream=stream,
                                                           bias=bias_k, beta=1.0), flush, stream, reps, warmup),
        "bwd_filter_with_bias_grads": _time_call(
            lambda: cg.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad, st, out=dw, workspace=ws_f, stream=stream,
                                         db_k=dbk, db_c=dbc), flush, stream, reps, warmup)}
    extra_ms = ex_ms["bwd_filter_with_bias_grads"] - op_ms["bwd_filter"]
    sum_bytes = (math.prod(pb.y_shape) + math.prod(pb.x_shape)) * pb.elem_bytes()  # dy and x read once
    fused = {"fwd_bias_addto_ms": round(ex_ms["fwd_bias_addto"], 5), "fwd_ms": round(op_ms["fwd"], 5),
             "bwd_filter_with_bias_grads_ms": round(ex_ms["bwd_filter_with_bias_grads"], 5),
             "bwd_filter_ms": round(op_ms["bwd_filter"], 5), "bias_grads_extra_ms": round(extra_ms, 5),
             "bias_grads_alg_gbs": round(sum_bytes / (extra_ms * 1e-3) / 1e9, 1) if extra_ms > 0 else None,
             "note": "bias gradients = channel sums of dy (per k) and x (per c); alg bytes = |dy| + |x|"}
    # dilation 2 on the same layer (pad 2 keeps P = H, Q = W, same FLOP)
    pad2 = (2 * pb.pad_h, 2 * pb.pad_w)
    wsz_d = cg.conv2d_workspace_size(2, (pb.N, pb.C, pb.H, pb.W, pb.K, pb.R, pb.S, pad2[0], pad2[1],
                                         pb.stride_h, pb.stride_w, pb.P, pb.Q), dt, (2, 2))
    ws_d = torch.empty(max(wsz_d, 16), dtype=torch.uint8, device=dev)
    dcalls = {"fwd": lambda: cg.conv2d_fwd(x, w, pad2, st, out=y, workspace=ws, stream=stream, dilation=2),
              "bwd_data": lambda: cg.conv2d_bwd_data(dy, w, (pb.H, pb.W), pad2, st, out=dx, workspace=ws,
                                                     stream=stream, dilation=2),
              "bwd_filter": lambda: cg.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad2, st, out=dw, workspace=ws_d,
                                                         stream=stream, dilation=2)}
    dilated = {}
    for op in OPS:
        ms = _time_call(dcalls[op], flush, stream, reps, warmup)
        dilated[op] = {"ms": round(ms, 5), "tflops": round(pb.flops() / (ms * 1e-3) / 1e12, 2)}
    dilated["note"] = "same layer with dilation 2 and pad 2 (P, Q unchanged, same FLOP)"
    # groups 2 on the same layer (two independent 32 -> 32 channel convolutions: half the FLOP)
    wg2 = w[:, : pb.C // 2].contiguous()
    wsz_g = max(cg.conv2d_workspace_size(op, pb.dims(), dt, (1, 1), 2) for op in range(3))
    ws_g = torch.empty(max(wsz_g, 16), dtype=torch.uint8, device=dev)
    dwg = torch.empty_like(wg2)
    gcalls = {"fwd": lambda: cg.conv2d_fwd(x, wg2, pad, st, out=y, workspace=ws_g, stream=stream, groups=2),
              "bwd_data": lambda: cg.conv2d_bwd_data(dy, wg2, (pb.H, pb.W), pad, st, out=dx, workspace=ws_g,
                                                     stream=stream, groups=2),
              "bwd_filter": lambda: cg.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad, st, out=dwg, workspace=ws_g,
                                                         stream=stream, groups=2)}
    grouped = {}
    for op in OPS:
        ms = _time_call(gcalls[op], flush, stream, reps, warmup)
        grouped[op] = {"ms": round(ms, 5), "tflops": round(pb.flops() / 2 / (ms * 1e-3) / 1e12, 2)}
    grouped["note"] = "same layer with groups 2 (C/2 -> K/2 per group, half the FLOP)"
    # depthwise on the same layer (groups = C = K = 64: one 3x3 filter per channel; memory
    # bound, so the rate is the op's algorithmic bytes against the HBM peak)
    wdw = w[:, :1].contiguous()
    wsz_w = max(cg.conv2d_workspace_size(op, pb.dims(), dt, (1, 1), pb.C) for op in range(3))
    ws_w = torch.empty(max(wsz_w, 16), dtype=torch.uint8, device=dev)
    dww = torch.empty_like(wdw)
    wcalls = {"fwd": lambda: cg.conv2d_fwd(x, wdw, pad, st, out=y, workspace=ws_w, stream=stream, groups=pb.C),
              "bwd_data": lambda: cg.conv2d_bwd_data(dy, wdw, (pb.H, pb.W), pad, st, out=dx, workspace=ws_w,
                                                     stream=stream, groups=pb.C),
              "bwd_filter": lambda: cg.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad, st, out=dww, workspace=ws_w,
                                                         stream=stream, groups=pb.C)}
    eb = pb.elem_bytes()
    io = {"fwd": math.prod(pb.x_shape) + math.prod(pb.y_shape), "bwd_data": math.prod(pb.y_shape) + math.prod(pb.x_shape),
          "bwd_filter": math.prod(pb.x_shape) + math.prod(pb.y_shape)}
    depthwise = {}
    for op in OPS:
        ms = _time_call(wcalls[op], flush, stream, reps, warmup)
        gbs = io[op] * eb / (ms * 1e-3) / 1e9
        depthwise[op] = {"ms": round(ms, 5), "alg_gbs": round(gbs, 1)}
    depthwise["note"] = ("same layer depthwise (groups = C = 64, filter 64 x 1 x 3 x 3); alg bytes = the two "
                         "activation tensors of the op (the filter is 2.3 KB)")
    cg.conv2d_device_status(stream)
    return fused, dilated, grouped, depthwise


def _e2e(c, flush, stream, nsteps):
    """End to end through the public API: pinned host inputs -> device -> three ops -> host
    results, every step.  Steps are pipelined over three streams with two device buffer sets:
    step i's input copies (stream s_in) overlap step i-1's ops (the compute stream) and step
    i-2's result copies (stream s_out); events order each buffer's reuse.  The timed region
    spans the first input copy to the last result copy.  Returns ms per step."""
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    pb = c["pb"]
    dev = c["x"].device
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    x, w, dy = c["host"]
    xh, wh, dyh = x.pin_memory(), w.pin_memory(), dy.pin_memory()
    ws = c["ws"]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = []
    for _ in range(2):
        bufs.append({"x": torch.empty_like(c["x"]), "w": torch.empty_like(c["w"]), "dy": torch.empty_like(c["dy"]),
                     "y": torch.empty_like(c["y"]), "dx": torch.empty_like(c["dx"]), "dw": torch.empty_like(c["dw"]),
                     "yh": torch.empty(pb.y_shape, dtype=x.dtype).pin_memory(),
                     "dxh": torch.empty(pb.x_shape, dtype=x.dtype).pin_memory(),
                     "dwh": torch.empty(pb.w_shape, dtype=x.dtype).pin_memory()})

    def run(n):
        ev_cmp = [torch.cuda.Event() for _ in range(n)]
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n):
            bb = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])  # step i-2's ops have read this input set
                bb["x"].copy_(xh, non_blocking=True)
                bb["w"].copy_(wh, non_blocking=True)
                bb["dy"].copy_(dyh, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i-2's results have been read back
            with torch.cuda.stream(stream):
                flush.zero_()
                cg.conv2d_fwd(bb["x"], bb["w"], pad, st, out=bb["y"], workspace=ws, stream=stream)
                cg.conv2d_bwd_data(bb["dy"], bb["w"], (pb.H, pb.W), pad, st, out=bb["dx"], workspace=ws,
                                   stream=stream)
                cg.conv2d_bwd_filter(bb["x"], bb["dy"], (pb.R, pb.S), pad, st, out=bb["dw"], workspace=ws,
                                     stream=stream)
                ev_cmp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                bb["yh"].copy_(bb["y"], non_blocking=True)
                bb["dxh"].copy_(bb["dx"], non_blocking=True)
                bb["dwh"].copy_(bb["dw"], non_blocking=True)
                ev_out[i].record(s_out)
        s_out.wait_event(ev_out[n - 1])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(2)  # warm-up of the streams and buffers
    return run(nsteps) / nsteps


def run_ours(args, rank, world):
    import torch
    import convolution_nchw_conv2d_gb300 as cg
    from convolution_nchw_conv2d_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    wl = W.WORKLOADS[args.workload]
    pb = wl.problem
    head = _device_case(wl, dev)
    for _ in range(args.warmup):
        for op in OPS:
            flush.zero_()
            _op_call(head, op, stream)
    cg.conv2d_device_status(stream)

    # ---- the timed steps: fwd + bwd_data + bwd_filter of the headline workload, L2 flushed
    # before every op outside its events
    K = args.steps
    evs = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K)] for op in OPS}
    sampler = ClockSampler(local)
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches0 = cg.conv2d_kernel_launches()
    t0 = time.time()
    for i in range(K):
        for op in OPS:
            flush.zero_()
            a, b = evs[op][i]
            a.record(stream)
            _op_call(head, op, stream)
            b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    launches = cg.conv2d_kernel_launches() - launches0
    clocks = sampler.stop(t0, t1)
    cg.conv2d_device_status(stream)
    op_ms = {op: sum(a.elapsed_time(b) for a, b in evs[op]) / K for op in OPS}
    step_ms = slowest_rank_ms(sum(op_ms.values()), world, dev)
    per_op, roof = _roofline_of(pb, op_ms, peaks)
    roof["traffic"] = ncu_traffic(wl.name, roof["kernel"])
    roof["peak_source"] = peaks["source"] + (" (bf16 x nominal tf32/bf16 ratio)" if pb.dtype == "f32" else "")

    # ---- every workload, each op timed alone the same way (the headline one included again)
    reps = max(1, min(args.config_reps, K))
    per_config = {}
    for name, wlc in W.WORKLOADS.items():
        c = head if name == wl.name else _device_case(wlc, dev)
        ms = {op: _time_call(lambda: _op_call(c, op, stream), flush, stream, reps, args.warmup) for op in OPS}
        cg.conv2d_device_status(stream)
        po, rf = _roofline_of(wlc.problem, ms, peaks)
        per_config[name] = {"shape": wlc.description, "dtype": "tf32" if wlc.problem.dtype == "f32" else "bf16",
                            "flop_per_op": wlc.problem.flops(), "alg_bytes_per_op": wlc.problem.alg_bytes("fwd"),
                            "per_op": po, "dominant": rf,
                            "step_tflops": round(3 * wlc.problem.flops() / (sum(ms.values()) * 1e-3) / 1e12, 2)}
        if c is not head:
            del c
    per_config["note"] = (f"each op timed alone ({reps} calls after {args.warmup} warm-up calls, L2 flushed before "
                          "every call); tensor peak TF32 for fp32 workloads, BF16 for bf16; the dominant op against "
                          "its roof (tensor or HBM by arithmetic intensity)")

    extras = {"fused_backward": _fused_backward(head, flush, stream, reps, args.warmup,
                                                {op: per_config[wl.name]["per_op"][op]["ms"] for op in OPS})}
    if "resnet3x3" in W.WORKLOADS:
        rc = head if wl.name == "resnet3x3" else _device_case(W.WORKLOADS["resnet3x3"], dev)
        rms = per_config["resnet3x3"]["per_op"]
        fused, dilated, grouped, depthwise = _extras_resnet(rc, flush, stream, reps, args.warmup,
                                                 {op: rms[op]["ms"] for op in OPS})
        extras.update({"fused_epilogue": fused, "dilation_2": dilated, "groups_2": grouped, "depthwise": depthwise})

    e2e_ms = _e2e(head, flush, stream, max(1, args.e2e_steps))
    esz = pb.elem_bytes()
    nx, ny, nw = (math.prod(pb.x_shape), math.prod(pb.y_shape), math.prod(pb.w_shape))
    flop = pb.flops()
    value = job_tflops(flop, len(OPS), world, step_ms)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if pb.dtype == "f32" else "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "shape": wl.description,
                   "N": pb.N, "C": pb.C, "H": pb.H, "W": pb.W, "K": pb.K, "R": pb.R, "S": pb.S,
                   "pad": [pb.pad_h, pb.pad_w], "stride": [pb.stride_h, pb.stride_w],
                   "step": "fwd + bwd_data + bwd_filter", "l2": "flushed before every op (2x L2 write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "per_op": per_op,
        "roofline": roof,
        "e2e": {"value": round(world * 3 * flop / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (nx + nw + ny) * esz, "d2h_bytes_per_step": (ny + nx + nw) * esz,
                "ms_per_step": round(e2e_ms, 4),
                "pipelined": "input copies, ops and result copies of consecutive steps overlap "
                             "on three streams (two device buffer sets)"},
        "gpu_launches": launches,
        "per_config": per_config,
        "clocks": clocks,
    }
    line.update(extras)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, seconds=12.0)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


# ------------------------------------------------------------------ oracle (CPU) arm
def _oracle_sample(wl, budget_s, rng_seed=0):
    """Time the fp64 oracle on random output elements of every op; returns (flop, seconds, desc)."""
    import numpy as np

    import oracle
    from convolution_nchw_conv2d_gb300 import workloads as W
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    xs, ws_, dys = (oracle._f64(t) for t in (x, w, dy))
    rng = np.random.default_rng(rng_seed)
    red = {"fwd": pb.C * pb.R * pb.S, "bwd_data": pb.K * pb.R * pb.S, "bwd_filter": pb.N * pb.P * pb.Q}
    sizes = {"fwd": math.prod(pb.y_shape), "bwd_data": math.prod(pb.x_shape), "bwd_filter": math.prod(pb.w_shape)}
    fns = {"fwd": (oracle.conv2d_fwd_at, xs, ws_), "bwd_data": (oracle.conv2d_bwd_data_at, dys, ws_),
           "bwd_filter": (oracle.conv2d_bwd_filter_at, xs, dys)}
    # calibrate: equal multiply-add budget per op
    macs_per_op = 2_000_000
    flop = 0
    t_all = 0.0
    counts = {}
    while True:
        flop = 0
        t0 = time.perf_counter()
        for op in OPS:
            n = max(1, min(sizes[op], macs_per_op // red[op]))
            counts[op] = n
            idx = rng.choice(sizes[op], size=n, replace=False)
            fn, a, b = fns[op]
            fn(a, b, pb.dims(), idx)
            flop += 2 * n * red[op]
        t_all = time.perf_counter() - t0
        full = all(counts[o] == sizes[o] for o in OPS)
        if t_all >= budget_s * 0.5 or full or macs_per_op > 10**12:
            break
        macs_per_op = int(macs_per_op * max(2.0, budget_s / max(t_all, 1e-3)))
    passes = 1
    if full and t_all < budget_s * 0.5:
        # every output of the step fits in the budget: repeat whole passes up to ~the budget
        extra = max(0, int(budget_s * 0.8 / max(t_all, 1e-3)) - 1)
        t0 = time.perf_counter()
        for _ in range(extra):
            for op in OPS:
                fn, a, b = fns[op]
                fn(a, b, pb.dims(), np.arange(sizes[op]))
        t_all += time.perf_counter() - t0
        flop *= 1 + extra
        passes += extra
    what = "every output" if full else f"{', '.join(f'{counts[o]} random {o} outputs' for o in OPS)}"
    desc = (f"{what} of the {wl.name} workload ({passes} pass{'es' if passes > 1 else ''}), each output a full "
            f"fp64 reduction (flop counted at 2*reduction length per output)")
    return flop, t_all, desc


def cpu_baseline(wl, seconds=12.0):
    import oracle
    flop, t, desc = _oracle_sample(wl, seconds)
    return {"value": flop / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": desc, "seconds": round(t, 3)}


def run_reference(args, rank, world):
    import oracle
    from convolution_nchw_conv2d_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    pb = wl.problem
    per_step = 2.0
    for _ in range(args.warmup):
        _oracle_sample(wl, 0.2)
    flops, secs = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        f, t, desc = _oracle_sample(wl, per_step)
        flops += f
        secs += t
    v = flops / secs / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "shape": wl.description, "step": "fwd + bwd_data + bwd_filter (sampled)"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.profile is not None:
        return run_profile(args)
    if args.impl == "reference":
        if rank != 0:
            return 0
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
