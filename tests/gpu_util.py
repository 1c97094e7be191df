"""Helpers for the GPU parity tests: move a seeded layer to the device, pack
its weights through the library, and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import bit_quantized_moe_q4_gb300 as moe

TOL_RMS = 2e-2  # max|gpu - oracle| <= 2e-2 * RMS(oracle output), per layer


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceLayer:
    """A LayerInputs on the GPU with packed weights."""

    def __init__(self, li, device="cuda", fmt=moe.MOE_Q4_CODES):
        self.li = li
        self.T, self.H, self.I, self.E, self.k = li.T, li.H, li.I, li.E, li.k
        self.x = bf16_tensor(li.x, device)
        self.wr = torch.from_numpy(li.wr).to(device)
        self.wgu = self._pack(li.gu_codes, li.gu_scales, device, fmt)
        self.wd = self._pack(li.d_codes, li.d_scales, device, fmt)

    @staticmethod
    def _pack(codes, scales, device, fmt):
        E, N, K = codes.shape
        if fmt == moe.MOE_Q4_CODES:
            c = torch.from_numpy(codes).to(device)
            s = torch.from_numpy(scales.view(np.int16)).to(device)
            out = moe.moe_q4_pack(c, s, E, N, K)
            del c, s
        else:
            import workloads
            b = torch.from_numpy(workloads.blocks18(codes, scales)).to(device)
            out = moe.moe_q4_pack(b, None, E, N, K, fmt=moe.MOE_Q4_BLOCK18)
            del b
        return out

    def prefill(self, out_fp32=True, debug=None, x=None, workspace=None):
        return moe.moe_q4_forward_prefill(self.x if x is None else x, self.wr, self.wgu, self.wd,
                                          self.I, self.k, out_fp32=out_fp32, debug=debug,
                                          workspace=workspace)

    def decode(self, out_fp32=True, debug=None, x=None, workspace=None):
        return moe.moe_w4a8_forward_decode(self.x if x is None else x, self.wr, self.wgu, self.wd,
                                           self.I, self.k, out_fp32=out_fp32, debug=debug,
                                           workspace=workspace)


def out_to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def assert_within_tol(gpu: np.ndarray, ref: np.ndarray, tol=TOL_RMS, what="output"):
    r = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.max(np.abs(gpu - ref)))
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    assert err <= tol * r, f"{what}: max|gpu-oracle| = {err:.4g} > {tol} * RMS {r:.4g}"
    return err / r
