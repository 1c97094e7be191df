"""The oracle's 8-bit weight path (the 8-bit setting of the companion page
"A Modern Multimodal Assistant on a 6 GB 2011 GPU: Stage-Validated, All-GPU
CUDA Inference for Fermi", Abstract), pinned to facts outside the oracle:

* a block worked by hand: d = fp16(amax / 127) exact at 2^-7, codes rounded
  half away from zero (0.5 d -> 1, -0.5 d -> -1, 1.5 d -> 2);
* the zero block (d = 0, all codes 0) and the code range (|q| <= 127);
* round trip within half a step;
* the integer group dots against an element-by-element Python loop;
* a 4-bit layer written as 8-bit codes (q - 8, same scales) gives the 4-bit
  decode layer bit for bit: the two paths differ only in where the offset
  8 is taken.
"""
import numpy as np

from oracle import moe_oracle as O


def test_q8_encode_hand_worked_block():
    d = 2.0 ** -7  # amax = 127 * 2^-7, so fp16(amax / 127) = 2^-7 exactly
    x = np.zeros(32)
    x[:6] = [127 * d, -0.5, 0.25, 0.5 * d, -0.5 * d, 1.5 * d]
    q, s = O.q8_encode(x[None, :])
    assert s.shape == (1, 1) and float(s[0, 0]) == d
    assert q.dtype == np.int8
    assert q[0, :6].tolist() == [127, -64, 32, 1, -1, 2]
    assert not q[0, 6:].any()


def test_q8_encode_zero_block_and_range():
    q, s = O.q8_encode(np.zeros((2, 64)))
    assert not q.any() and not s.astype(np.float64).any()
    rng = np.random.default_rng(5)
    w = rng.standard_normal((16, 256)) * rng.uniform(1e-3, 10, (16, 1))
    q, s = O.q8_encode(w)
    assert np.abs(q.astype(np.int64)).max() <= 127
    # the block maximum maps to +-127 (or +-126 when fp16 rounded d up)
    qb = np.abs(q.astype(np.int64)).reshape(16, 8, 32).max(axis=-1)
    assert (qb >= 126).all()


def test_q8_round_trip_within_half_a_step():
    rng = np.random.default_rng(6)
    w = rng.standard_normal((8, 128))
    q, s = O.q8_encode(w)
    back = O.q8_dequant(q, s)
    d = np.repeat(s.astype(np.float64), 32, axis=-1)
    assert (np.abs(back - w) <= 0.5 * d * (1 + 1e-3) + 1e-12).all()


def test_group_dots8_against_a_loop():
    rng = np.random.default_rng(7)
    codes = rng.integers(-127, 128, (3, 64)).astype(np.int8)
    qa = rng.integers(-127, 128, 64)
    G = O.group_dots8(codes, qa)
    for r in range(3):
        for g in range(2):
            want = 0
            for i in range(32):
                want += int(codes[r, 32 * g + i]) * int(qa[32 * g + i])
            assert G[r, g] == want


def test_q4_layer_as_8bit_codes_is_the_same_layer():
    import workloads as W
    li = W.make_layer("q8pin", 3, 128, 128, 4, 2, seed=9, wr_std=0.1)
    out4, st4 = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k,
                             keep_dots=True, prenorm=True)
    gu8 = (li.gu_codes.astype(np.int16) - 8).astype(np.int8)
    d8 = (li.d_codes.astype(np.int16) - 8).astype(np.int8)
    out8, st8 = O.moe_decode(li.x, li.wr, gu8, li.gu_scales, d8, li.d_scales, li.k,
                             keep_dots=True, prenorm=True, wbits=8)
    assert np.array_equal(out4, out8)
    for key in st4["dots_gu"]:
        assert np.array_equal(st4["dots_gu"][key], st8["dots_gu"][key])
        assert np.array_equal(st4["dots_d"][key], st8["dots_d"][key])
