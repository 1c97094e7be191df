"""Benchmark of the 4-bit MoE expert-FFN layer on one GB300 (or N replicas).

Default workload: the batch-1 W4A8 decode layer (T=1, H=2048, I=768, E=128,
top-8), timed as CUDA-graph replays of a chain of 16 layers whose packed
weights are distinct copies, so each step touches ~360 MB (> the 129 MB L2).
The same line carries the T=4 and T=16 decode layers and the T=2048 prefill
layer (one call per step; its 340 MB of packed weights exceed L2).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer prefill tokens/s and decode µs/token; % of HBM / tensor roofline"
DECODE_LAYERS = 16          # distinct weight copies per decode step
GU_BYTES_PER_EXPERT = 2 * 768 * 2048 * 18 // 32   # packed gate/up bytes of one expert
D_BYTES_PER_EXPERT = 2048 * 768 * 18 // 32        # packed down bytes of one expert
# DRAM bytes (read + write) per launch from one ncu capture of each kernel as
# it is in this tree: the decode expert kernel (T=1) and the prefill expert
# GEMMs (T=2048).  Set to None when the kernel changes before a new capture.
NCU_TRAFFIC_DECODE_EXPERTS_T1 = 22_540_288
NCU_TRAFFIC_PREFILL_EXPERTS = None  # not yet captured for the single-launch expert GEMMs
KERNELS_PER_DECODE_LAYER = 2   # layer (router, top-k, buckets, x codes, gate/up, down); combine
KERNELS_PER_PREFILL_LAYER = 7  # W_r split, router GEMM, top-k + chunk counts, bucket scan, scatter, expert GEMMs, combine


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
def _device_layer(li, torch, moe, device):
    x = torch.from_numpy(li.x.view(np.int16)).to(device).view(torch.bfloat16)
    wr = torch.from_numpy(li.wr).to(device)

    def pack(codes, scales):
        E, N, K = codes.shape
        c = torch.from_numpy(codes).to(device)
        s = torch.from_numpy(scales.view(np.int16)).to(device)
        out = moe.moe_q4_pack(c, s, E, N, K)
        del c, s
        return out

    return x, wr, pack(li.gu_codes, li.gu_scales), pack(li.d_codes, li.d_scales)


def bench_decode(T, steps, warmup, torch, moe, device, barrier):
    import workloads
    li = workloads.decode(T)
    x, wr, wgu, wd = _device_layer(li, torch, moe, device)
    L = DECODE_LAYERS
    layers = [(wr.clone(), wgu.clone(), wd.clone()) for _ in range(L)]
    del wgu, wd
    outs = [torch.empty((T, li.H), dtype=torch.float32, device=device) for _ in range(L)]
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, li.H, li.I, li.E, li.k),
                     dtype=torch.uint8, device=device)
    stages = moe.StageEvents()
    # distinct experts this token batch touches (from the library's own routing)
    idx, _ = moe.moe_route_topk(x, wr, li.k)
    distinct = int(torch.unique(idx).numel())

    def run_layers():
        for l, (wr_l, wgu_l, wd_l) in enumerate(layers):
            moe.moe_w4a8_forward_decode(x, wr_l, wgu_l, wd_l, li.I, li.k, out=outs[l],
                                        workspace=ws, debug=stages.debug if l == L - 1 else None)

    run_layers()  # load modules outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        run_layers()
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_step = t0.elapsed_time(t1) / steps
    barrier()
    # per-kernel durations of the last layer of each replay (stage events)
    ex_ms, cb_ms = [], []
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        ex_ms.append(stages.ms(0, 1))
        cb_ms.append(stages.ms(5, 6))
    # end to end: pinned host x in, graph, last layer's output back to the host
    x_host = torch.empty((T, li.H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    out_host = torch.empty((T, li.H), dtype=torch.float32, pin_memory=True)
    for _ in range(3):
        x.copy_(x_host, non_blocking=True)
        g.replay()
        out_host.copy_(outs[-1], non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        x.copy_(x_host, non_blocking=True)
        g.replay()
        out_host.copy_(outs[-1], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / steps
    gu_bytes = distinct * GU_BYTES_PER_EXPERT
    dn_bytes = distinct * D_BYTES_PER_EXPERT
    layer_bytes = gu_bytes + dn_bytes + li.E * li.H * 4 + T * li.H * (2 + 4)
    res = {
        "T": T, "layers_per_step": L, "ms_per_step": ms_step,
        "us_per_token": ms_step * 1e3 / (L * T),
        "us_per_layer": ms_step * 1e3 / L,
        "distinct_experts": distinct,
        "algorithmic_bytes_per_layer": layer_bytes,
        "layer_gbs": layer_bytes / (ms_step / L * 1e-3) / 1e9,
        # the layer kernel: routing, then gate/up and down
        "experts_us": statistics.mean(ex_ms) * 1e3, "combine_us": statistics.mean(cb_ms) * 1e3,
        "gateup_bytes": gu_bytes, "down_bytes": dn_bytes, "router_bytes": li.E * li.H * 4,
        "e2e_us_per_token": e2e_ms * 1e3 / (L * T),
        "h2d_bytes_per_step": T * li.H * 2, "d2h_bytes_per_step": T * li.H * 4,
        "kernels_per_step": L * KERNELS_PER_DECODE_LAYER,
    }
    res["experts_gbs"] = (gu_bytes + dn_bytes + li.E * li.H * 4) / (res["experts_us"] * 1e-6) / 1e9
    del layers, outs, ws, g
    torch.cuda.empty_cache()
    return res


def bench_prefill(name, steps, warmup, torch, moe, device, barrier):
    import workloads
    li = workloads.CONFIGS[name]()
    x, wr, wgu, wd = _device_layer(li, torch, moe, device)
    T, H, I, E, k = li.T, li.H, li.I, li.E, li.k
    out = torch.empty((T, H), dtype=torch.float32, device=device)
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL, T, H, I, E, k),
                     dtype=torch.uint8, device=device)
    stages = moe.StageEvents()

    def call(dbg=None):
        moe.moe_q4_forward_prefill(x, wr, wgu, wd, I, k, out=out, workspace=ws, debug=dbg)

    for _ in range(max(warmup, 3)):
        call()
    torch.cuda.synchronize()
    barrier()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    barrier()
    per = {"route": [], "bucket": [], "experts": [], "combine": []}
    for _ in range(steps):
        call(stages.debug)
        torch.cuda.synchronize()
        per["route"].append(stages.ms(0, 1))
        per["bucket"].append(stages.ms(1, 2))
        per["experts"].append(stages.ms(3, 5))  # gate/up and down: one launch
        per["combine"].append(stages.ms(5, 6))
    us = {kk: statistics.mean(v) * 1e3 for kk, v in per.items()}
    gu_flop = 2.0 * T * k * H * 2 * I
    dn_flop = 2.0 * T * k * I * H
    # e2e: pinned host x in, one layer, output back
    x_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    out_host = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
    for _ in range(3):
        x.copy_(x_host, non_blocking=True)
        call()
        out_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        x.copy_(x_host, non_blocking=True)
        call()
        out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / steps
    counts = None
    res = {
        "workload": name, "T": T, "ms_per_layer": ms, "tokens_per_s": T / (ms * 1e-3),
        "layer_tflops": (gu_flop + dn_flop + 2.0 * T * E * H) / (ms * 1e-3) / 1e12,
        "stage_us": us,
        "experts_tflops": (gu_flop + dn_flop) / (us["experts"] * 1e-6) / 1e12,
        "gateup_flop": gu_flop, "down_flop": dn_flop,
        "e2e_tokens_per_s": T / (e2e_ms * 1e-3),
        "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4,
    }
    del x, wr, wgu, wd, out, ws
    torch.cuda.empty_cache()
    return res


def bench_prefill_stack(steps, warmup, torch, moe, device, barrier):
    """The 40-layer pre-norm stack (T=4096, H=2048, I=768, E=256, k=8, fresh
    counter-generated Q4_0 weights per layer, 27.2 GB resident): one step runs
    all layers, bf16 between them; reports ms per layer."""
    import workloads as W
    S = W.STACK
    L, T, H, I, E, k = S["L"], S["T"], S["H"], S["I"], S["E"], S["k"]
    chunk = 32
    layers = []
    for l in range(L):
        wgu = torch.empty(moe.moe_q4_packed_bytes(E, 2 * I, H), dtype=torch.uint8, device=device)
        wd = torch.empty(moe.moe_q4_packed_bytes(E, H, I), dtype=torch.uint8, device=device)
        per_gu, per_d = wgu.numel() // E, wd.numel() // E
        for e0 in range(0, E, chunk):
            gc, gs, dc, ds = W.stacked_experts_torch(l, e0, e0 + chunk, device)
            moe.moe_q4_pack(gc, gs.view(torch.int16), chunk, 2 * I, H,
                            out=wgu[e0 * per_gu:(e0 + chunk) * per_gu])
            moe.moe_q4_pack(dc, ds.view(torch.int16), chunk, H, I,
                            out=wd[e0 * per_d:(e0 + chunk) * per_d])
            del gc, gs, dc, ds
        layers.append((torch.from_numpy(W.stacked_router(l)).to(device), wgu, wd))
    x0 = torch.from_numpy(W.stacked_x().view(np.int16)).to(device).view(torch.bfloat16)
    bufs = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(2)]
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL, T, H, I, E, k),
                     dtype=torch.uint8, device=device)

    def step():
        cur = x0
        for l, (wr, wgu, wd) in enumerate(layers):
            nxt = bufs[l % 2]
            moe.moe_q4_forward_prefill(cur, wr, wgu, wd, I, k, out=nxt, out_fp32=False,
                                       workspace=ws, prenorm=True)
            cur = nxt

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_stack = t0.elapsed_time(t1) / steps
    flop = 2.0 * T * k * 3 * H * I
    res = {"workload": "stacked", "layers": L, "T": T, "E": E, "ms_per_stack": ms_stack,
           "ms_per_layer": ms_stack / L, "tokens_per_s": T / (ms_stack * 1e-3),
           "expert_tflops": flop * L / (ms_stack * 1e-3) / 1e12}
    del layers, x0, bufs, ws
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------
def _cpu_usage(fn):
    """Runs fn(); returns (wall seconds, effective cores = cpu time / wall)."""
    c0, w0 = time.process_time(), time.perf_counter()
    fn()
    c1, w1 = time.process_time(), time.perf_counter()
    wall = w1 - w0
    return wall, (c1 - c0) / wall if wall > 0 else 1.0


def cpu_baseline_decode(T=1, budget_s=12.0):
    """The oracle's W4A8 decode of T=1 tokens, repeated for about budget_s."""
    import workloads
    from oracle import moe_oracle as O
    li = workloads.decode(T)
    n = [0]

    def run():
        t_end = time.perf_counter() + budget_s
        while True:
            O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
            n[0] += 1
            if time.perf_counter() > t_end:
                break

    wall, cores = _cpu_usage(run)
    return {"value": wall * 1e6 / (n[0] * T), "unit": "µs/token", "cores": round(cores, 1),
            "kind": "oracle",
            "sample": f"{n[0]} oracle decode layer call(s) of T={T} (H=2048, I=768, E=128, k=8), "
                      f"{wall:.1f} s wall"}


def cpu_baseline_prefill(ntok=16):
    import workloads
    from oracle import moe_oracle as O
    li = workloads.prefill()
    toks = np.arange(ntok)
    wall, cores = _cpu_usage(lambda: O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales,
                                                   li.d_codes, li.d_scales, li.k, tokens=toks))
    return {"value": ntok / wall, "unit": "tokens/s", "cores": round(cores, 1), "kind": "oracle",
            "sample": f"{ntok} of the 2048 prefill tokens through the oracle, {wall:.1f} s wall"}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one decode layer call
    on one token (a bounded sample of the decode workload)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import workloads
    from oracle import moe_oracle as O
    li = workloads.decode(1)

    def step():
        O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)

    for _ in range(args.warmup):
        step()
    times = []
    c0, w0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        s0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - s0)
    wall = time.perf_counter() - w0
    cores = (time.process_time() - c0) / wall
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "µs/token",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64/int64", "data": "synthetic",
        "config": {"workload": "decode W4A8 MoE layer, T=1, H=2048, I=768, E=128, top-8",
                   "parallelism": "single process (CPU oracle)"},
        "cpu_baseline": {"value": us, "unit": "µs/token", "cores": round(cores, 1),
                         "kind": "oracle", "sample": f"{args.steps} oracle decode calls, T=1"},
        "e2e": {"value": us, "unit": "µs/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def rank_ops(dist, world, device):
    """barrier() and max_over_ranks(v) over the default process group (no-ops
    for a single process); `device` holds the reduction buffer (the GPU under
    NCCL, the CPU under gloo)."""
    import torch

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        if world == 1:
            return float(v)
        t = torch.tensor([float(v)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def decode_value(ms_step_max, layers_per_step, world):
    """Whole-job µs per token: the slowest rank's step time over the tokens
    all ranks decoded in it (one token per layer per rank)."""
    return ms_step_max * 1e3 / (layers_per_step * world)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--only", choices=["decode", "prefill"], default=None,
                    help="run one workload only (short profiling runs)")
    ap.add_argument("--decode-tokens", type=str, default="1,4,16")
    ap.add_argument("--prefill-workload", choices=["prefill", "skewed", "stacked"],
                    default="prefill",
                    help="with --only prefill: the T=2048 layer, the Zipf-skewed T=10240 "
                         "layer or the 40-layer E=256 stack")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.prefill_workload != "prefill" and args.only != "prefill":
        ap.error("--prefill-workload other than prefill needs --only prefill")

    import torch
    import torch.distributed as dist

    import bit_quantized_moe_q4_gb300 as moe
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    moe.build()
    moe.load_library()

    barrier, max_over_ranks = rank_ops(dist, world, device)

    peaks = load_peaks()
    warm = max(args.warmup, 3)
    dec_T = [int(t) for t in args.decode_tokens.split(",")] if args.only != "prefill" else []
    if args.only != "prefill" and 1 not in dec_T:
        dec_T = [1] + dec_T
    with ClockSampler(local) as clk:
        dec = {T: bench_decode(T, args.steps, warm, torch, moe, device, barrier) for T in dec_T}
        if args.no_prefill or args.only == "decode":
            pre = None
        elif args.prefill_workload == "stacked":
            pre = bench_prefill_stack(min(args.steps, 10), warm, torch, moe, device, barrier)
        else:
            pre = bench_prefill(args.prefill_workload, args.steps, warm, torch, moe, device,
                                barrier)
    if args.only == "prefill":
        print(json.dumps({"prefill": pre, "clocks": clk.summary()}))
        return 0
    clocks = clk.summary()
    status = moe.moe_get_device_status()

    d1 = dec[1]
    ms_step = max_over_ranks(d1["ms_per_step"])
    value = decode_value(ms_step, d1["layers_per_step"], world)
    e2e_ms = max_over_ranks(d1["e2e_us_per_token"] * d1["layers_per_step"] / 1e3)
    roof_gbs = d1["experts_gbs"]
    line = {
        "metric": METRIC, "value": value, "unit": "µs/token", "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": ms_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights x int8 activations (int32 group dots, fp32 scales)",
        "data": "synthetic",
        "config": {
            "workload": "decode W4A8 MoE layer: T=1, H=2048, I=768, E=128, top-8 "
                        "(batch-1 decode config); step = CUDA-graph replay of 16 layers with "
                        "distinct weight copies",
            "l2": "inputs larger than L2: each step touches ~360 MB of distinct weights",
            "parallelism": "replicas only" if world > 1 else "single GPU",
        },
        "roofline": {"bound": "hbm", "kernel": "decode_experts_kernel", "achieved": roof_gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": roof_gbs / peaks["hbm_gbs"], "traffic": NCU_TRAFFIC_DECODE_EXPERTS_T1,
                     "peak_source": peaks["source"],
                     "algorithmic_bytes_per_launch": d1["gateup_bytes"] + d1["down_bytes"] +
                                                     d1["router_bytes"],
                     "launch_us": d1["experts_us"]},
        "e2e": {"value": e2e_ms * 1e3 / (d1["layers_per_step"] * world), "unit": "µs/token",
                "h2d_bytes_per_step": d1["h2d_bytes_per_step"],
                "d2h_bytes_per_step": d1["d2h_bytes_per_step"]},
        "gpu_launches": args.steps * d1["kernels_per_step"],
        "clocks": clocks,
        "decode": {f"T{T}": r for T, r in dec.items()},
        "device_status": status,
    }
    if pre is not None:
        line["prefill"] = pre
        line["prefill_roofline"] = {
            "bound": "tensor", "kernel": "grouped_q4_gemm_kernel (gate/up, then down)",
            "achieved": pre["experts_tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": pre["experts_tflops"] / peaks["bf16_tflops"],
            "traffic": NCU_TRAFFIC_PREFILL_EXPERTS,
            "peak_source": peaks["source"]}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(1)
        if pre is not None:
            line["prefill"]["cpu_baseline"] = cpu_baseline_prefill(16)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
