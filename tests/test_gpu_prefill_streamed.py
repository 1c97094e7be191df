"""GPU: the streamed prefill stack (moe_q4_forward_prefill_stack_streamed)
through the C ABI: the experts stay in pinned host memory and reach the GPU
layer by layer, overlapped with the layers' compute.

The page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU",
Methodology 1 "Prefill (GPU)": the experts live in host RAM and move to the
GPU one layer at a time.  Streaming changes only where the weights come from,
so the output must equal the chained single-layer calls on device-resident
weights bit for bit; those calls are pinned to the oracle by the layer tests.

Cases: three small pre-norm layers (bf16 and fp32 last outputs), one layer,
two layers of the full-size prefill shape, a CUDA-graph capture of the call,
and the refusal of weights in pageable host memory.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer  # noqa: E402


def _layers(n, T, H, I, E, k, seed0):
    return [DeviceLayer(W.make_layer("streamed", T, H, I, E, k, seed=seed0 + l, wr_std=1.0 / np.sqrt(H)))
            for l in range(n)]


def _chain(x, layers, I, k, out_fp32_last):
    cur = x
    for l, d in enumerate(layers):
        last = l == len(layers) - 1
        cur = moe.moe_q4_forward_prefill(cur, d.wr, d.wgu, d.wd, I, k, out_fp32=out_fp32_last and last,
                                         prenorm=True)
    return cur


def _host(layers):
    # (router rows on the device, packed experts in pinned host memory)
    return [(d.wr, d.wgu.cpu().pin_memory(), d.wd.cpu().pin_memory()) for d in layers]


def _bits(t):
    if t.dtype == torch.float32:
        return t.cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("n,out_fp32", [(3, False), (3, True), (1, True)])
def test_streamed_equals_device_resident_chain(n, out_fp32):
    T, H, I, E, k = 96, 256, 128, 8, 2
    layers = _layers(n, T, H, I, E, k, seed0=40)
    x = layers[0].x
    ref = _chain(x, layers, I, k, out_fp32)
    out = moe.moe_q4_forward_prefill_stack_streamed(x, _host(layers), I, k, out_fp32=out_fp32)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert np.array_equal(_bits(out), _bits(ref))


def test_streamed_full_size_two_layers():
    li = [W.prefill(seed=s) for s in (2, 3)]
    layers = [DeviceLayer(l) for l in li]
    d0 = layers[0]
    x = d0.x
    ref = _chain(x, layers, d0.I, d0.k, False)
    out = moe.moe_q4_forward_prefill_stack_streamed(x, _host(layers), d0.I, d0.k, out_fp32=False)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))


def test_streamed_graph_replay():
    T, H, I, E, k = 64, 256, 128, 8, 2
    layers = _layers(4, T, H, I, E, k, seed0=60)
    host = _host(layers)
    x = layers[0].x
    ref = _chain(x, layers, I, k, False)
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL_STREAMED, T, H, I, E, k),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_q4_forward_prefill_stack_streamed(x, host, I, k, out=out, out_fp32=False, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        moe.moe_q4_forward_prefill_stack_streamed(x, host, I, k, out=out, out_fp32=False, workspace=ws)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))


def test_streamed_refuses_pageable_host_memory():
    T, H, I, E, k = 16, 256, 128, 8, 2
    d = _layers(1, T, H, I, E, k, seed0=80)[0]
    pageable = d.wgu.cpu()  # not page-locked
    lib = moe.load_library()
    arr = lambda p: (ctypes.c_void_p * 1)(p)
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL_STREAMED, T, H, I, E, k),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    rc = lib.moe_q4_forward_prefill_stack_streamed(
        ctypes.c_void_p(d.x.data_ptr()), 1, arr(d.wr.data_ptr()), arr(pageable.data_ptr()),
        arr(d.wd.cpu().pin_memory().data_ptr()), T, H, I, E, k, moe.MOE_STACKED_PRENORM,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert b"pinned" in lib.moe_last_error_string()
