"""GPU Q4_0 encoder (moe_q4_quantize) against the oracle's encode, bit for bit.

The rule (page "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011
GPU", Methodology 2 "Quantization", read as the Q4_0 family's usual encoder):
per block of 32, m = the largest-magnitude element (first on a tie, sign
kept), d = fp16(m / -8), q = min(15, max(0, floor(x / d + 8.5))) against the
stored d, d = 0 -> q = 8.  Checked on the hand-worked blocks (negative scale,
magnitude tie, clamp, zero block), on blocks whose elements sit exactly on a
rounding boundary x = (n - 8.5) d and one fp32 ulp to either side, on random
fp32 and bf16 tensors, and in both output formats.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")


def _gpu_encode(w32: np.ndarray, fmt=None, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(w32, np.float32)).cuda()
    if bf16:
        t = t.to(torch.bfloat16)
    if fmt is None:
        c, s = moe.moe_q4_quantize(t)
        return c.cpu().numpy(), s.cpu().numpy()
    return moe.moe_q4_quantize(t, fmt=fmt).cpu().numpy()


def _check_equal(w32):
    c, s = _gpu_encode(w32)
    qo, do = O.q4_encode(np.asarray(w32, np.float64))
    assert np.array_equal(s.view(np.uint16), do.view(np.uint16)), "scales differ"
    assert np.array_equal(c, qo), f"{int((c != qo).sum())} codes differ"
    return c, s


def test_encode_hand_worked_blocks():
    x = np.zeros((4, 32), np.float32)
    x[0, :5] = [-2.0, 1.0, 0.3, 1.9, 0.0]   # d = 0.25: codes 0, 12, 9, 16 -> 15, 8
    x[1, :2] = [2.0, -1.0]                  # d = -0.25: codes 0, 12
    x[2, 0], x[2, 5] = 1.0, -1.0            # magnitude tie: the first sets d = -0.125
    c, s = _check_equal(x)                  # row 3: zero block, d = 0, codes 8
    assert s.astype(np.float64)[:, 0].tolist() == [0.25, -0.25, -0.125, 0.0]
    assert c[0, :5].tolist() == [0, 12, 9, 15, 8] and np.all(c[0, 5:] == 8)
    assert c[1, :2].tolist() == [0, 12]
    assert c[2, 0] == 0 and c[2, 5] == 15
    assert np.all(c[3] == 8)


def test_encode_exact_rounding_boundaries():
    # d = fp16(m / -8) with m = -8 * 0.0371 (not a power of two); elements at
    # x = (n - 8.5) d exactly (floor(x/d + 8.5) = n) and one fp32 ulp either
    # side (n - 1 or n, depending on the side and the sign of d).
    rows = []
    for m in (-8 * 0.0371, 8 * 0.0371, -3.3, 5.5e-3):
        d = float(np.float16(m / -8.0))
        for n in range(1, 16):
            t = np.float32((n - 8.5) * d)
            row = np.zeros(32, np.float32)
            row[0] = m
            row[1] = t
            row[2] = np.nextafter(t, np.float32(np.inf))
            row[3] = np.nextafter(t, np.float32(-np.inf))
            rows.append(row)
    _check_equal(np.stack(rows))


@pytest.mark.parametrize("bf16", [False, True])
def test_encode_random_tensors(bf16):
    rng = np.random.default_rng(17)
    parts = [rng.standard_normal((64, 1024)),
             rng.standard_normal((64, 1024)) * 1e-3,
             rng.standard_normal((64, 1024)) * 300.0,
             rng.uniform(-1, 1, (64, 1024)) ** 7]        # many tiny values
    w = np.concatenate(parts).astype(np.float32)
    if bf16:
        w = O.bf16_bits_to_f32(workloads.f32_to_bf16_bits(w))
    c, s = _gpu_encode(w, bf16=bf16)
    qo, do = O.q4_encode(w.astype(np.float64))
    assert np.array_equal(s.view(np.uint16), do.view(np.uint16))
    assert np.array_equal(c, qo)


def test_encode_blocks18_and_pack_roundtrip():
    rng = np.random.default_rng(3)
    E, N, K = 2, 128, 256
    w = (rng.standard_normal((E, N, K)) * 0.05).astype(np.float32)
    blocks = _gpu_encode(w, fmt=moe.MOE_Q4_BLOCK18)
    qo, do = O.q4_encode(w.astype(np.float64))
    assert np.array_equal(blocks, workloads.blocks18(qo, do))
    # the encoder's output feeds moe_q4_pack: both formats give one layout
    c, s = moe.moe_q4_quantize(torch.from_numpy(w).cuda())
    p1 = moe.moe_q4_pack(c, s.view(torch.int16), E, N, K)
    p2 = moe.moe_q4_pack(torch.from_numpy(blocks).cuda(), None, E, N, K, fmt=moe.MOE_Q4_BLOCK18)
    assert torch.equal(p1, p2)


def test_encode_empty_and_shape_errors():
    w = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    c, s = moe.moe_q4_quantize(w)
    assert c.shape == (0, 64) and s.shape == (0, 2)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_q4_quantize(torch.zeros((4, 40), dtype=torch.float32, device="cuda"))
    assert ei.value.code == moe.MOE_ERR_SHAPE
