"""The allocation-free decode entry point (moe_w4a8_forward_decode_noalloc).

It serves callers that cannot allocate device memory — components hosted by
an application that owns all device memory, or decode loops that must not call
cudaMalloc — by running the decode layer on a fixed scratch array inside the
library.  Checked here through the C ABI: two calls in a row agree with the
workspace-taking entry point within the layer tolerance, and a shape whose
scratch would not fit is rejected.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer, TOL_RMS, out_to_f64  # noqa: E402


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


def test_noalloc_rejects_scratch_overflow():
    # T = 32, H = 4096, I = 1536, E = 256, k = 8 needs ~4.8 MB of scratch, more
    # than the 4 MiB array; the call is refused before any weight is read, so
    # small placeholder weight buffers suffice.
    T, H, I, E, k = 32, 4096, 1536, 256, 8
    assert moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, H, I, E, k) > moe.MOE_NOALLOC_SCRATCH_BYTES
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    placeholder = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_w4a8_forward_decode_noalloc(x, wr, placeholder, placeholder, I, k)
    assert ei.value.code == moe.MOE_ERR_WORKSPACE
    assert "scratch" in str(ei.value)
