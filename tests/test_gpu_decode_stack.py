"""GPU: the stacked decode entry (moe_w4a8_forward_decode_stack) through the
C ABI, against the chain of single-layer decode calls, bit for bit.

The per-token decode loop of the page "A 35B Hybrid-Attention Mixture-of-
Experts Model on a 6GB 2011 GPU" (Methodology 1, "Decode (CPU)"): every
generated token runs through every layer's experts.  The stack runs the same
kernels as the single-layer call, one call enqueueing all layers (layer
l + 1 reading layer l's output rounded to bf16), so its output must equal the
chained calls' bits; the single-layer path is pinned to the oracle by the
layer tests and along the oracle's own chain (the decode-chain test), and one
case here also follows the oracle's chain directly.

Cases: the first 8 layers of the stacked workload (E = 256) at T = 1, 4
(clustered layer kernel), 16 and 32 (the task kernel and its T > 16
variant); three E = 128 layers; fp32 and bf16 last outputs, with and without
the pre-norm; a stack of one; repeated calls, a garbage-filled workspace and
a captured graph replay.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer  # noqa: E402
from test_gpu_stacked import _gpu_layer  # noqa: E402

L8 = 8


@pytest.fixture(scope="module")
def stack8():
    return [_gpu_layer(l, "cuda") for l in range(L8)]


def _x(T, H, seed=7):
    xb = W.stacked_x()[:T] if H == W.STACK["H"] and T <= 32 else None
    if xb is None:
        rng = np.random.default_rng(seed)
        xb = W.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to("cuda").view(torch.bfloat16)


def _chain(x, layers, I, k, prenorm, out_fp32_last, ws):
    cur = x
    for l, (wr, wgu, wd) in enumerate(layers):
        last = l == len(layers) - 1
        cur = moe.moe_w4a8_forward_decode(cur, wr, wgu, wd, I, k, out_fp32=out_fp32_last and last,
                                          workspace=ws, prenorm=prenorm)
    return cur


def _bits(t):
    if t.dtype == torch.float32:
        return t.cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _ws(T, H, I, E, k, fill=None):
    n = moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, H, I, E, k)
    if fill is None:
        return torch.empty(n, dtype=torch.uint8, device="cuda")
    return torch.full((n,), fill, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("T", [1, 4, 16, 32])
def test_stack_equals_chained_calls_E256(stack8, T):
    S = W.STACK
    H, I, E, k = S["H"], S["I"], S["E"], S["k"]
    x = _x(T, H)
    ref = _chain(x, stack8, I, k, True, False, _ws(T, H, I, E, k))
    out = moe.moe_w4a8_forward_decode_stack(x, stack8, I, k, out_fp32=False, prenorm=True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert np.array_equal(_bits(out), _bits(ref))


@pytest.fixture(scope="module")
def stack128():
    # three E = 128 layers of the decode shape, distinct weights
    return [DeviceLayer(W.make_layer("stack128", 16, 2048, 768, 128, 8, seed=11 + l,
                                     wr_std=1.0 / np.sqrt(2048)))
            for l in range(3)]


@pytest.mark.parametrize("T,prenorm,out_fp32", [(16, True, True), (4, False, False), (1, False, True)])
def test_stack_equals_chained_calls_E128(stack128, T, prenorm, out_fp32):
    layers = [(d.wr, d.wgu, d.wd) for d in stack128]
    H, I, E, k = 2048, 768, 128, 8
    x = stack128[0].x[:T].contiguous()
    ref = _chain(x, layers, I, k, prenorm, out_fp32, _ws(T, H, I, E, k))
    out = moe.moe_w4a8_forward_decode_stack(x, layers, I, k, out_fp32=out_fp32, prenorm=prenorm)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert out.dtype == (torch.float32 if out_fp32 else torch.bfloat16)
    assert np.array_equal(_bits(out), _bits(ref))


def test_stack_of_one_is_the_layer(stack128):
    d = stack128[1]
    x = d.x[:4].contiguous()
    ref = moe.moe_w4a8_forward_decode(x, d.wr, d.wgu, d.wd, d.I, d.k, out_fp32=True)
    out = moe.moe_w4a8_forward_decode_stack(x, [(d.wr, d.wgu, d.wd)], d.I, d.k, out_fp32=True,
                                            prenorm=False)
    assert np.array_equal(_bits(out), _bits(ref))


def test_stack_follows_the_oracle_chain(stack8):
    # one token through 4 layers: the stack against the oracle's own chain
    # (the oracle never sees a GPU value), each layer's tolerance compounded
    # only through the oracle's inputs
    S = W.STACK
    H, I, E, k, L = S["H"], S["I"], S["E"], S["k"], 4
    xb = W.stacked_x()[:1]
    outs = []
    for l in range(L):
        out, st = O.moe_decode(xb, *W.stacked_layer_lazy(l), k, prenorm=True)
        xb = O.f64_to_bf16_bits(out)
        outs.append(out)
    x = _x(1, H)
    got = moe.moe_w4a8_forward_decode_stack(x, stack8[:L], I, k, out_fp32=True, prenorm=True)
    g = got.cpu().numpy().astype(np.float64)
    o = outs[-1]
    # the GPU's layer inputs are its own bf16 outputs, so the layers' errors
    # add up: allow L times the per-layer bound
    assert np.all(np.abs(g - o) <= L * (2e-2 * O.rms(o)) + np.abs(o) * 2.0 ** -7)


def test_stack_repeatable_graph_and_garbage_workspace(stack128):
    layers = [(d.wr, d.wgu, d.wd) for d in stack128]
    H, I, E, k, T = 2048, 768, 128, 8, 4
    x = stack128[2].x[:T].contiguous()
    ws = _ws(T, H, I, E, k, fill=0x7F)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_w4a8_forward_decode_stack(x, layers, I, k, out=out, out_fp32=False, workspace=ws)
    first = _bits(out).copy()
    for _ in range(3):
        moe.moe_w4a8_forward_decode_stack(x, layers, I, k, out=out, out_fp32=False, workspace=ws)
        assert np.array_equal(_bits(out), first)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        moe.moe_w4a8_forward_decode_stack(x, layers, I, k, out=out, out_fp32=False, workspace=ws)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert np.array_equal(_bits(out), first)
