"""Benchmark of the 4-bit MoE expert-FFN layer on one GB300 (or N replicas).

Default workload: the batch-1 W4A8 decode layer (T=1, H=2048, I=768, E=128,
top-8) in its decode loop: a step is one CUDA-graph replay of a chain of 16
pre-norm layers whose packed weights are distinct copies, layer l + 1
decoding layer l's bf16 output, so each step touches ~360 MB (> the 129 MB
L2).  The same line carries the T=4 and T=16 chains, the T=2048 prefill
layer, the Zipf-skewed T=10240 prefill layer and the 40-layer E=256 prefill
stack (27 GB of weights resident).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead, on all host cores.
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
STREAMED_LAYERS = 8         # layers of the stacked prefill timed with host-resident experts
GU_BYTES_PER_EXPERT = 2 * 768 * 2048 * 18 // 32   # packed gate/up bytes of one expert
D_BYTES_PER_EXPERT = 2048 * 768 * 18 // 32        # packed down bytes of one expert
# DRAM bytes (read + write) per launch from one ncu capture of each kernel as
# it is in this tree: the decode prep and layer kernels (T=1) and the prefill
# expert GEMMs (T=2048).  Set to None when a kernel changes before a new
# capture.
# DRAM bytes (read + write) of one decode layer at T=1: the prep, clustered
# and combine kernels, averages of 10 launches each under ncu (1.093 + 21.330 + 0.406 MB)
NCU_TRAFFIC_DECODE_LAYER_T1 = 22_828_262
NCU_TRAFFIC_PREFILL_EXPERTS = 384_733_696  # dram read + write, ncu, one launch at T=2048
# kernels of one decode layer: prep (logits, x codes) and, for T <= 16, the
# clustered expert kernel and the combine kernel; else the task kernel (top-k,
# buckets, experts, combine)


def kernels_per_decode_layer(T):
    return 3 if T <= 16 else 2

DECODE_WORKLOAD = ("decode W4A8 MoE layer: T=1, H=2048, I=768, E=128, top-8 (batch-1 decode "
                   "config), in a chain of 16 pre-norm layers with distinct weight copies, "
                   "each layer decoding the previous one's bf16 output")
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


def bench_decode(T, steps, warmup, torch, moe, device, barrier, L=DECODE_LAYERS, w8=True):
    """A chain of L pre-norm decode layers (distinct weight copies) in one CUDA
    graph: layer l + 1 decodes layer l's bf16 output."""
    import workloads
    li = workloads.decode(T)
    x, wr, wgu, wd = _device_layer(li, torch, moe, device)
    layers = [(wr.clone(), wgu.clone(), wd.clone()) for _ in range(L)]
    del wr, wgu, wd
    outs = [torch.empty((T, li.H), dtype=torch.bfloat16, device=device) for _ in range(L)]
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, li.H, li.I, li.E, li.k),
                     dtype=torch.uint8, device=device)
    idx = [torch.empty((T, li.k), dtype=torch.int32, device=device) for _ in range(L)]
    dbgs = [moe.MoeDebug(topk_idx=b.data_ptr()) for b in idx]

    def run_chain(debug=False):
        cur = x
        for l, (wr_l, wgu_l, wd_l) in enumerate(layers):
            moe.moe_w4a8_forward_decode(cur, wr_l, wgu_l, wd_l, li.I, li.k, out=outs[l],
                                        out_fp32=False, workspace=ws, prenorm=True,
                                        debug=dbgs[l] if debug else None)
            cur = outs[l]

    run_chain(debug=True)  # loads the modules outside the capture; routing per layer
    torch.cuda.synchronize()
    distinct = [int(torch.unique(b).numel()) for b in idx]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        run_chain()
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
    # end to end: each step takes the chain's input from pinned host memory
    # and returns its output there (T tokens in, T tokens out per step)
    x_host = torch.empty((T, li.H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    out_host = torch.empty((T, li.H), dtype=torch.bfloat16, pin_memory=True)
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
    # the same L layers from one call (moe_w4a8_forward_decode_stack): its
    # output must carry the chain's bits
    out_stack = torch.empty((T, li.H), dtype=torch.bfloat16, device=device)

    def run_stack():
        moe.moe_w4a8_forward_decode_stack(x, layers, li.I, li.k, out=out_stack, out_fp32=False,
                                          workspace=ws, prenorm=True)

    run_stack()
    run_chain()
    torch.cuda.synchronize()
    stack_same = bool(torch.equal(out_stack.view(torch.int16), outs[-1].view(torch.int16)))
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, capture_error_mode="relaxed"):
        run_stack()
    for _ in range(max(warmup, 3)):
        gs.replay()
    torch.cuda.synchronize()
    barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(steps):
        gs.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    ms_stack = s0.elapsed_time(s1) / steps
    barrier()
    s0.record(stream)
    for _ in range(steps):
        x.copy_(x_host, non_blocking=True)
        gs.replay()
        out_host.copy_(out_stack, non_blocking=True)
    s1.record(stream)
    torch.cuda.synchronize()
    e2e_stack_ms = s0.elapsed_time(s1) / steps
    expert_bytes = GU_BYTES_PER_EXPERT + D_BYTES_PER_EXPERT
    # algorithmic bytes of each layer: its touched experts' packed weights,
    # the router, x in and the output out (bf16)
    layer_bytes = [d * expert_bytes + li.E * li.H * 4 + T * li.H * (2 + 2) for d in distinct]
    us_layer = ms_step * 1e3 / L
    res = {
        "T": T, "layers_per_step": L, "chained": True, "prenorm": True, "ms_per_step": ms_step,
        "us_per_token": us_layer / T, "us_per_layer": us_layer,
        "distinct_experts_per_layer": distinct,
        "algorithmic_bytes_per_layer": statistics.mean(layer_bytes),
        "layer_gbs": statistics.mean(layer_bytes) / (us_layer * 1e-6) / 1e9,
        "e2e_us_per_token": e2e_ms * 1e3 / (L * T),
        "h2d_bytes_per_step": T * li.H * 2, "d2h_bytes_per_step": T * li.H * 2,
        "kernels_per_step": L * kernels_per_decode_layer(T),
        "stack": {
            "entry": "moe_w4a8_forward_decode_stack (one call: the L layers' kernels, chained by PDL)",
            "equals_chain_bits": stack_same, "ms_per_step": ms_stack,
            "us_per_layer": ms_stack * 1e3 / L, "us_per_token": ms_stack * 1e3 / (L * T),
            "layer_gbs": statistics.mean(layer_bytes) / (ms_stack * 1e3 / L * 1e-6) / 1e9,
            "e2e_us_per_token": e2e_stack_ms * 1e3 / (L * T),
            "kernels_per_step": L * kernels_per_decode_layer(T),
        },
    }
    if w8 and T <= moe.MOE_W8_DECODE_MAX_T:
        res["w8"] = _decode_w8_chain(li, x, [l[0] for l in layers], outs[-1], distinct, ws, steps,
                                     warmup, torch, moe, device, barrier)
    del layers, outs, ws, g, gs
    torch.cuda.empty_cache()
    return res


def _decode_w8_chain(li, x, wrs, ref_out, distinct, ws, steps, warmup, torch, moe, device, barrier):
    """The same chain on the 8-bit weight path: each layer's 4-bit codes
    written as int8 (q - 8) with the same scales, packed as 8-bit tiles, so
    the layers move 34/18 of the 4-bit bytes and must return the 4-bit
    chain's bits."""
    T = li.T

    def pack8(codes, scales):
        E, N, K = codes.shape
        c = torch.from_numpy((codes.astype(np.int16) - 8).astype(np.int8)).to(device)
        s = torch.from_numpy(scales.view(np.int16)).to(device)
        out = moe.moe_q8_pack(c, s, E, N, K)
        del c, s
        return out

    wgu8, wd8 = pack8(li.gu_codes, li.gu_scales), pack8(li.d_codes, li.d_scales)
    layers8 = [(wr, wgu8.clone(), wd8.clone()) for wr in wrs]
    del wgu8, wd8
    outs8 = [torch.empty((T, li.H), dtype=torch.bfloat16, device=device) for _ in wrs]

    def run():
        cur = x
        for l, (wr_l, wgu_l, wd_l) in enumerate(layers8):
            moe.moe_w8a8_forward_decode(cur, wr_l, wgu_l, wd_l, li.I, li.k, out=outs8[l],
                                        out_fp32=False, workspace=ws, prenorm=True)
            cur = outs8[l]

    run()
    torch.cuda.synchronize()
    same = bool(torch.equal(outs8[-1].view(torch.int16), ref_out.view(torch.int16)))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        run()
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
    ms = t0.elapsed_time(t1) / steps
    L = len(wrs)
    expert_bytes8 = (GU_BYTES_PER_EXPERT + D_BYTES_PER_EXPERT) * 34 // 18
    layer_bytes = [d * expert_bytes8 + li.E * li.H * 4 + T * li.H * (2 + 2) for d in distinct]
    us_layer = ms * 1e3 / L
    res = {
        "entry": "moe_w8a8_forward_decode (8-bit tiles: 32 int8 codes + one fp16 scale per group)",
        "equals_4bit_chain_bits": same, "ms_per_step": ms, "us_per_layer": us_layer,
        "us_per_token": us_layer / T, "algorithmic_bytes_per_layer": statistics.mean(layer_bytes),
        "layer_gbs": statistics.mean(layer_bytes) / (us_layer * 1e-6) / 1e9,
    }
    del layers8, outs8, g
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
    # the first NS layers with their experts in pinned host memory,
    # streamed to the GPU layer by layer (moe_q4_forward_prefill_stack_streamed)
    NS = STREAMED_LAYERS
    gu_b, d_b = layers[0][1].numel(), layers[0][2].numel()
    pinned = torch.empty(NS * (gu_b + d_b), dtype=torch.uint8, pin_memory=True)
    host = []
    for l in range(NS):
        o = l * (gu_b + d_b)
        pinned[o:o + gu_b].copy_(layers[l][1])
        pinned[o + gu_b:o + gu_b + d_b].copy_(layers[l][2])
        host.append((layers[l][0], pinned[o:o + gu_b], pinned[o + gu_b:o + gu_b + d_b]))
    sws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL_STREAMED, T, H, I, E, k),
                      dtype=torch.uint8, device=device)
    sout = torch.empty((T, H), dtype=torch.bfloat16, device=device)

    def streamed():
        moe.moe_q4_forward_prefill_stack_streamed(x0, host, I, k, out=sout, out_fp32=False,
                                                  workspace=sws, prenorm=True)

    streamed()
    cur = x0  # the same layers on device-resident weights, for the bits check
    for l in range(NS):
        nxt = bufs[l % 2]
        moe.moe_q4_forward_prefill(cur, layers[l][0], layers[l][1], layers[l][2], I, k, out=nxt,
                                   out_fp32=False, workspace=ws, prenorm=True)
        cur = nxt
    torch.cuda.synchronize()
    same = bool(torch.equal(sout.view(torch.int16), cur.view(torch.int16)))
    barrier()
    nst = max(2, steps // 4)
    t0.record(stream)
    for _ in range(nst):
        streamed()
    t1.record(stream)
    torch.cuda.synchronize()
    ms_str = t0.elapsed_time(t1) / nst
    # the link's copy rate: one layer's experts copied alone from pinned
    # host memory, the same bytes the streamed stack moves per layer
    gd = torch.empty(gu_b + d_b, dtype=torch.uint8, device=device)
    src = host[0][1]
    dst = gd[: src.numel()]
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
        gd[src.numel(): src.numel() + host[0][2].numel()].copy_(host[0][2], non_blocking=True)
    t1.record(stream)
    torch.cuda.synchronize()
    copy_gbs = 3 * (gu_b + d_b) / (t0.elapsed_time(t1) * 1e-3) / 1e9
    del gd
    res["streamed"] = {
        "entry": "moe_q4_forward_prefill_stack_streamed (experts in pinned host memory, copied "
                 "layer by layer on a copy stream, overlapped with the layers' kernels)",
        "layers": NS, "ms_per_layer": ms_str / NS,
        "expert_bytes_per_layer": gu_b + d_b,
        "h2d_gbs": (gu_b + d_b) * NS / (ms_str * 1e-3) / 1e9,
        "plain_copy_gbs": copy_gbs,
        "copy_frac": (gu_b + d_b) * NS / (ms_str * 1e-3) / 1e9 / copy_gbs,
        "device_resident_ms_per_layer": ms_stack / L,
        "equals_device_chain_bits": same,
    }
    del layers, x0, bufs, ws, host, pinned, sws, sout
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------
def cpu_info():
    """CPU model and the cores this process may run on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"model": model or "unknown", "cores": int(cores)}


def _oracle_decode_worker(args):
    """One worker of the CPU baseline: the oracle's W4A8 decode of the T=1
    workload, repeated until `budget_s` has passed (after one untimed call).
    Returns (calls, seconds)."""
    budget_s, = args
    import workloads
    from oracle import moe_oracle as O
    li = workloads.decode(1)
    call = lambda: O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes,  # noqa: E731
                                li.d_scales, li.k)
    call()
    n, t0 = 0, time.perf_counter()
    while True:
        call()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            return n, time.perf_counter() - t0


def _oracle_prefill_worker(args):
    """The oracle's prefill layer on a subset of the T=2048 workload's tokens;
    returns the seconds it took (after loading the inputs)."""
    tokens, = args
    import workloads
    from oracle import moe_oracle as O
    li = workloads.prefill()
    t0 = time.perf_counter()
    O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k,
                  tokens=np.asarray(tokens))
    return time.perf_counter() - t0


def _pool(n):
    import concurrent.futures
    import multiprocessing
    return concurrent.futures.ProcessPoolExecutor(n, mp_context=multiprocessing.get_context("spawn"))


def cpu_baseline_decode(budget_s=8.0, workers=None):
    """The oracle's decode layer (T=1) on every host core: one process per core,
    each repeating the call; µs per token = wall time / calls."""
    info = cpu_info()
    n = workers or info["cores"]
    with _pool(n) as ex:
        res = list(ex.map(_oracle_decode_worker, [(budget_s,)] * n))
    calls = sum(c for c, _ in res)
    wall = max(t for _, t in res)
    return {"value": wall * 1e6 / calls, "unit": "µs/token", "cores": n, "kind": "oracle",
            "cpu_model": info["model"],
            "sample": f"{calls} oracle decode layer calls of T=1 (H=2048, I=768, E=128, k=8) "
                      f"in {n} processes over {wall:.1f} s"}


def cpu_baseline_prefill(tokens_per_worker=2, workers=None):
    """The oracle's prefill layer on a bounded sample of the T=2048 workload's
    tokens, split over every host core; tokens/s = sampled tokens / wall."""
    info = cpu_info()
    n = workers or info["cores"]
    chunks = [list(range(i * tokens_per_worker, (i + 1) * tokens_per_worker)) for i in range(n)]
    with _pool(n) as ex:
        secs = list(ex.map(_oracle_prefill_worker, [(c,) for c in chunks]))
    ntok = n * tokens_per_worker
    wall = max(secs)
    return {"value": ntok / wall, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "cpu_model": info["model"],
            "sample": f"{ntok} of the 2048 prefill tokens ({tokens_per_worker} per process, "
                      f"{n} processes), {wall:.1f} s"}


def run_reference(args):
    """The CPU oracle as the reference arm, on every host core: each step is one
    decode layer call on one token in each of the processes (a bounded
    sample of the T=1 decode workload); µs per token = step wall / processes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    info = cpu_info()
    n = info["cores"]
    with _pool(n) as ex:
        list(ex.map(_oracle_decode_worker, [(0.0,)] * n))  # spawn and load every worker
        for _ in range(args.warmup):
            list(ex.map(_oracle_decode_worker, [(0.0,)] * n))
        times = []
        for _ in range(args.steps):
            s0 = time.perf_counter()
            calls = sum(c for c, _ in ex.map(_oracle_decode_worker, [(0.0,)] * n))
            times.append((time.perf_counter() - s0) / calls)
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "µs/token",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us * n / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64/int64", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "parallelism": f"{n} CPU processes (oracle)"},
        "cpu_baseline": {"value": us, "unit": "µs/token", "cores": n, "kind": "oracle",
                         "cpu_model": info["model"],
                         "sample": f"{args.steps} steps of {n} concurrent oracle decode calls, T=1 "
                                   "(each process loads the workload once, untimed)"},
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


def prefill_roofline(pre, peaks, traffic=None):
    """The expert GEMMs' throughput against the dense bf16/fp16 peak."""
    return {"bound": "tensor", "kernel": "grouped_q4_gemm_kernel (gate/up, then down)",
            "achieved": pre["experts_tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": pre["experts_tflops"] / peaks["bf16_tflops"], "traffic": traffic,
            "peak_source": peaks["source"] + " (burst)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-stack", action="store_true",
                    help="leave the 40-layer prefill stack (27 GB of weights) out")
    ap.add_argument("--only", choices=["decode", "prefill"], default=None,
                    help="run one workload only (short profiling runs)")
    ap.add_argument("--decode-tokens", type=str, default="1,4,16")
    ap.add_argument("--no-w8", action="store_true",
                    help="leave the 8-bit-weight decode chain out")
    ap.add_argument("--decode-layers", type=int, default=DECODE_LAYERS,
                    help="layers in the decode chain (fewer: smaller profiling runs)")
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
    if args.only is None and 1 not in dec_T:
        dec_T = [1] + dec_T  # the headline is the T=1 chain
    pre = skew = stack = None
    with ClockSampler(local) as clk:
        dec = {T: bench_decode(T, args.steps, warm, torch, moe, device, barrier,
                               L=args.decode_layers, w8=not args.no_w8) for T in dec_T}
        if args.only == "prefill":
            if args.prefill_workload == "stacked":
                pre = bench_prefill_stack(min(args.steps, 10), warm, torch, moe, device, barrier)
            else:
                pre = bench_prefill(args.prefill_workload, args.steps, warm, torch, moe, device,
                                    barrier)
        elif not (args.no_prefill or args.only == "decode"):
            pre = bench_prefill("prefill", args.steps, warm, torch, moe, device, barrier)
            skew = bench_prefill("skewed", min(args.steps, 20), warm, torch, moe, device, barrier)
            if not args.no_stack:
                stack = bench_prefill_stack(3, 3, torch, moe, device, barrier)
    if args.only == "prefill":
        print(json.dumps({"prefill": pre, "clocks": clk.summary()}))
        return 0
    if args.only == "decode":
        print(json.dumps({"decode": {f"T{T}": r for T, r in dec.items()}, "clocks": clk.summary(),
                          "device_status": moe.moe_get_device_status()}))
        return 0
    clocks = clk.summary()
    status = moe.moe_get_device_status()

    d1 = dec[1]
    ms_step = max_over_ranks(d1["ms_per_step"])
    value = decode_value(ms_step, d1["layers_per_step"], world)
    e2e_ms = max_over_ranks(d1["e2e_us_per_token"] * d1["layers_per_step"] / 1e3)
    # the decode layer (prep + layer kernel) as it runs in the graph: the
    # per-layer replay time, an upper bound on the two kernels' duration
    us_layer = ms_step * 1e3 / d1["layers_per_step"]
    roof_gbs = d1["algorithmic_bytes_per_layer"] / (us_layer * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "µs/token", "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": ms_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights x int8 activations (int32 group dots, fp32 scales)",
        "data": "synthetic",
        "config": {
            "workload": DECODE_WORKLOAD if args.decode_layers == DECODE_LAYERS else
            DECODE_WORKLOAD.replace("16", str(args.decode_layers)),
            "l2": "inputs larger than L2: each step touches ~360 MB of distinct weights",
            "parallelism": "replicas only" if world > 1 else "single GPU",
        },
        "roofline": {"bound": "hbm",
                     "kernel": "decode_prep_kernel + decode_cluster_kernel + decode_combine_kernel",
                     "achieved": roof_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": roof_gbs / peaks["hbm_gbs"], "traffic": NCU_TRAFFIC_DECODE_LAYER_T1,
                     "peak_source": peaks["source"] + " (copy)",
                     "algorithmic_bytes_per_launch": d1["algorithmic_bytes_per_layer"],
                     "launch_us": us_layer,
                     "duration": "per-layer CUDA-graph replay time of the 16-layer chain"},
        "e2e": {"value": e2e_ms * 1e3 / (d1["layers_per_step"] * world), "unit": "µs/token",
                "h2d_bytes_per_step": d1["h2d_bytes_per_step"],
                "d2h_bytes_per_step": d1["d2h_bytes_per_step"],
                "step": "the token's input copied in from pinned host memory, the 16-layer "
                        "chain, its output copied back"},
        "gpu_launches": args.steps * d1["kernels_per_step"],
        "clocks": clocks,
        "decode": {f"T{T}": r for T, r in dec.items()},
        "device_status": status,
    }
    for T, r in dec.items():
        r["hbm_frac"] = r["layer_gbs"] / peaks["hbm_gbs"]
    if pre is not None:
        line["prefill"] = pre
        line["prefill_roofline"] = prefill_roofline(pre, peaks, NCU_TRAFFIC_PREFILL_EXPERTS)
    if skew is not None:
        line["prefill_skewed"] = skew
        line["prefill_skewed"]["roofline"] = prefill_roofline(skew, peaks)
    if stack is not None:
        line["prefill_stacked"] = stack
        line["prefill_stacked"]["roofline"] = {
            "bound": "tensor", "kernel": "the whole pre-norm layer (40 per step)",
            "achieved": stack["expert_tflops"], "peak": peaks["bf16_tflops_sustained"],
            "unit": "TFLOP/s", "frac": stack["expert_tflops"] / peaks["bf16_tflops_sustained"],
            "traffic": None, "peak_source": peaks["source"] + " (sustained)"}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode()
        if pre is not None:
            line["prefill"]["cpu_baseline"] = cpu_baseline_prefill()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
