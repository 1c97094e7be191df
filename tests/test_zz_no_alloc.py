"""The allocation-free decode entry point (moe_w4a8_forward_decode_noalloc).

It serves callers that cannot allocate device memory — components hosted by
an application that owns all device memory, or decode loops that must not call
cudaMalloc — by running the decode layer on a fixed scratch array inside the
library.  Checked here through the C ABI: two calls in a row agree with the
workspace-taking entry point within the layer tolerance; calls of different
shapes share the array (each call clears what it synchronises on), also when
a CUDA graph captured at one shape is replayed after an eager call of
another; the pre-norm flag passes through; a shape whose scratch would not
fit is rejected.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer, TOL_RMS, assert_within_tol, out_to_f64  # noqa: E402


def _check_against_workspace_entry(li):
    dl = DeviceLayer(li)
    ref = out_to_f64(dl.decode())
    r = float(np.sqrt(np.mean(ref * ref)))
    for _ in range(2):  # two calls in a row share the same scratch array
        out = torch.full((li.T, li.H), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_w4a8_forward_decode_noalloc(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k, out=out)
        got = out_to_f64(out)
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref))) <= TOL_RMS * r


def test_noalloc_decode_tiny():
    li = workloads.tiny()
    li.T = 16
    li.x = li.x[:16].copy()
    _check_against_workspace_entry(li)


def test_noalloc_decode_full_size():
    _check_against_workspace_entry(workloads.decode(4))


def _tokens(li, T):
    li.T = T
    li.x = li.x[:T].copy()
    return li


def test_noalloc_mixed_token_counts():
    # T = 1, 4, 1 in a row on the one array: the scratch offsets move with T,
    # so each call must clear its own counters.
    base = workloads.decode(16)
    layers = {T: DeviceLayer(_tokens(workloads.decode(16), T)) for T in (1, 4)}
    refs = {T: out_to_f64(dl.decode()) for T, dl in layers.items()}
    for T in (1, 4, 1, 4, 1):
        dl = layers[T]
        out = moe.moe_w4a8_forward_decode_noalloc(dl.x, dl.wr, dl.wgu, dl.wd, base.I, base.k)
        assert np.array_equal(out_to_f64(out), refs[T])  # fixed summation order: same bits
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0


def test_noalloc_graph_replay_after_other_shape():
    li1 = _tokens(workloads.decode(16), 1)
    li16 = workloads.decode(16)
    d1, d16 = DeviceLayer(li1), DeviceLayer(li16)
    ref1, _ = O.moe_decode(li1.x, li1.wr, li1.gu_codes, li1.gu_scales, li1.d_codes,
                           li1.d_scales, li1.k)
    ws_ref1 = out_to_f64(d1.decode())
    ws_ref16 = out_to_f64(d16.decode())
    out1 = torch.empty((1, li1.H), dtype=torch.float32, device="cuda")
    call1 = lambda: moe.moe_w4a8_forward_decode_noalloc(  # noqa: E731
        d1.x, d1.wr, d1.wgu, d1.wd, li1.I, li1.k, out=out1)
    call1()  # first call on the device: before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        call1()
    out16 = moe.moe_w4a8_forward_decode_noalloc(d16.x, d16.wr, d16.wgu, d16.wd, li16.I, li16.k)
    out1.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert np.array_equal(out_to_f64(out16), ws_ref16)
    assert np.array_equal(out_to_f64(out1), ws_ref1)
    assert_within_tol(out_to_f64(out1), ref1)


def test_noalloc_prenorm_flag():
    li = _tokens(workloads.decode(16), 4)
    dl = DeviceLayer(li)
    ref = out_to_f64(moe.moe_w4a8_forward_decode(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k,
                                                 prenorm=True))
    out = moe.moe_w4a8_forward_decode_noalloc(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k,
                                              prenorm=True)
    assert np.array_equal(out_to_f64(out), ref)


def test_noalloc_rejects_scratch_overflow():
    # T = 16, H = 4096, I = 2048, E = 256, k = 16 fits the on-chip staging but
    # needs ~8.7 MiB of scratch, more than the 8 MiB array; the call is refused
    # before any weight is read, so small placeholder weight buffers suffice.
    T, H, I, E, k = 16, 4096, 2048, 256, 16
    assert moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, H, I, E, k) > moe.MOE_NOALLOC_SCRATCH_BYTES
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    placeholder = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a8_forward_decode_noalloc(x, wr, placeholder, placeholder, I, k)
    assert ei.value.code == moe.MOE_ERR_WORKSPACE
    assert "scratch" in str(ei.value)
