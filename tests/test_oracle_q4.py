"""Pins for the oracle's Q4_0-family weight format (CPU only).

Each expected value below is worked by hand from the definition of the
Q4_0 family named on the page "A 35B Hybrid-Attention Mixture-of-Experts
Model on a 6GB 2011 GPU" (Methodology 2, "Quantization": group-wise symmetric
4-bit weights): blocks of 32 codes q in 0..15 sharing one fp16 scale d, with
w = d * (q - 8).  The derivations are written next to the numbers.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
import workloads


def _block(vals, fill=8):
    b = np.full(32, fill, dtype=np.uint8)
    b[: len(vals)] = vals
    return b


def test_dequant_worked_example_two_blocks():
    # Row of 64 codes = two blocks.  Block 0: d = 0.25 (fp16 0x3400);
    # Block 1: d = -0.5 (fp16 0xB800).
    codes = np.concatenate([_block([0, 8, 15, 1]), _block([0, 15, 9])])[None, :]
    scales = np.array([[0x3400, 0xB800]], dtype=np.uint16).view(np.float16)
    w = O.q4_dequant(codes, scales)
    # block 0: 0.25*(0-8) = -2, 0.25*(8-8) = 0, 0.25*(15-8) = 1.75, 0.25*(1-8) = -1.75
    assert w[0, :4].tolist() == [-2.0, 0.0, 1.75, -1.75]
    assert np.all(w[0, 4:32] == 0.0)
    # block 1: -0.5*(0-8) = 4, -0.5*(15-8) = -3.5, -0.5*(9-8) = -0.5
    assert w[0, 32:35].tolist() == [4.0, -3.5, -0.5]
    assert np.all(w[0, 35:] == 0.0)


def test_dequant_batched_rows_use_their_own_scales():
    # Two experts x two rows, one block each, codes all 15 (q - 8 = 7).
    codes = np.full((2, 2, 32), 15, dtype=np.uint8)
    scales = np.array([[[1.0], [2.0]], [[0.5], [4.0]]], dtype=np.float16)
    w = O.q4_dequant(codes, scales)
    assert w[0, 0, 0] == 7.0 and w[0, 1, 5] == 14.0
    assert w[1, 0, 31] == 3.5 and w[1, 1, 0] == 28.0


def test_encode_worked_example():
    # Largest magnitude is -2.0, so d = fp16(-2 / -8) = 0.25.
    x = np.zeros(32)
    x[:5] = [-2.0, 1.0, 0.3, 1.9, 0.0]
    q, d = O.q4_encode(x[None, :])
    assert d.astype(np.float64).ravel().tolist() == [0.25]
    # floor(-2/0.25 + 8.5) = floor(0.5) = 0; floor(4 + 8.5) = 12;
    # floor(1.2 + 8.5) = 9; floor(7.6 + 8.5) = 16 -> clamped to 15; floor(8.5) = 8
    assert q[0, :5].tolist() == [0, 12, 9, 15, 8]
    assert np.all(q[0, 5:] == 8)
    # decoded: -2, 1.0, 0.25, 1.75, 0
    assert O.q4_dequant(q, d)[0, :5].tolist() == [-2.0, 1.0, 0.25, 1.75, 0.0]


def test_encode_negative_scale_and_ties_and_zero_block():
    # Largest magnitude +2.0 -> d = -0.25; 2/-0.25 + 8.5 = 0.5 -> q = 0 -> w = -0.25*(-8) = 2.
    x = np.zeros((3, 32))
    x[0, :2] = [2.0, -1.0]          # -1/-0.25 + 8.5 = 12.5 -> 12 -> w = -0.25*4 = -1
    x[1, 0], x[1, 5] = 1.0, -1.0    # magnitude tie: the first (+1.0) sets d = -0.125
    q, d = O.q4_encode(x)
    assert d.astype(np.float64).ravel().tolist() == [-0.25, -0.125, 0.0]
    assert q[0, :2].tolist() == [0, 12]
    assert O.q4_dequant(q[:1], d[:1])[0, :2].tolist() == [2.0, -1.0]
    assert q[1, 0] == 0 and q[1, 5] == 16 - 1  # -1/-0.125 + 8.5 = 16.5 -> 16 -> 15
    assert np.all(q[2] == 8)                   # zero block: d = 0, q = 8
    assert np.all(O.q4_dequant(q[2:], d[2:]) == 0.0)


def test_encode_roundtrip_error_bound():
    # Away from the clamp, decode(encode(x)) is within |d|/2 of x (plus the
    # fp16 rounding of d acting on |x|/|d| <= 8 steps).
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256))
    q, d = O.q4_encode(x)
    w = O.q4_dequant(q, d)
    dd = np.repeat(np.abs(d.astype(np.float64)), 32, axis=-1)
    unclamped = q != 15
    err = np.abs(w - x)
    assert np.all(err[unclamped] <= 0.5 * dd[unclamped] * (1 + 1e-3) + 1e-12)
    # the clamp only costs one extra step at the block maximum's mirror
    assert np.all(err <= 1.5 * dd + 1e-12)


def test_blocks18_hand_built():
    # scale 0x3400 = 0.25, little-endian bytes 00 34; byte 0 = 0xF0 -> element 0 = 0,
    # element 16 = 15; byte 1 = 0x18 -> element 1 = 8, element 17 = 1; others 0x88.
    blk = np.full(18, 0x88, dtype=np.uint8)
    blk[0], blk[1] = 0x00, 0x34
    blk[2], blk[3] = 0xF0, 0x18
    codes, scales = O.q4_from_blocks18(blk[None, :])
    assert scales.astype(np.float64).tolist() == [0.25]
    expect = [8] * 32
    expect[0], expect[16], expect[1], expect[17] = 0, 15, 8, 1
    assert codes.reshape(-1).tolist() == expect


def test_blocks18_generator_roundtrip():
    li = workloads.tiny()
    blocks = workloads.blocks18(li.gu_codes[:2], li.gu_scales[:2])
    codes, scales = O.q4_from_blocks18(blocks)
    assert np.array_equal(codes, li.gu_codes[:2])
    assert np.array_equal(scales.view(np.uint16), li.gu_scales[:2].view(np.uint16))


def test_generated_codes_and_scales_in_range():
    li = workloads.tiny()
    assert li.gu_codes.max() == 15 and li.gu_codes.min() == 0
    s = li.d_scales.astype(np.float64)
    assert s.min() >= 0.0049 and s.max() <= 0.0201
    # codes are uniform: each value about 1/16 of the total
    hist = np.bincount(li.gu_codes.ravel(), minlength=16) / li.gu_codes.size
    assert np.all(np.abs(hist - 1 / 16) < 0.01)
