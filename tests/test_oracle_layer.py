"""Pins for the oracle's whole-layer evaluations (CPU only).

The layer is the MoE expert FFN of the page "A 35B Hybrid-Attention
Mixture-of-Experts Model on a 6GB 2011 GPU" (Methodology 1: grouped 4-bit GEMM
over routed experts in prefill, W4A8 integer kernel in decode; Methodology 2:
Q4_0-family weights, 8-bit decode activations), read as: router top-k with
softmax weights, SwiGLU expert FFN (gate, up, down), weighted combine plus
residual.  The hand-computed case below fixes signs, the q - 8 offset, which
projection goes through silu, the block-to-scale mapping and the residual.
"""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O
import workloads


def _bits(v):
    return workloads.f32_to_bf16_bits(np.asarray(v, np.float32))


def _hand_layer(x_val, k=1):
    """H = 64, I = 32, E = 2.  Expert 0: gate codes 9 (q-8 = 1) with block
    scales 1/32 and 1/64; up codes 12 (q-8 = 4), scales 1/64; down rows
    alternate codes 7 (q-8 = -1) and 10 (q-8 = 2), scale 1/2.  Expert 1 has
    zero scales.  Router: expert 0 weights 1/64 (exact in fp32), expert 1 weights 0."""
    H, I, E = 64, 32, 2
    x = _bits(np.full((1, H), x_val))
    wr = np.zeros((E, H), np.float32)
    wr[0] = 1 / 64
    gu_codes = np.zeros((E, 2 * I, H), np.uint8)
    gu_scales = np.zeros((E, 2 * I, H // 32), np.float16)
    gu_codes[0, :I] = 9
    gu_scales[0, :I, 0] = 1 / 32
    gu_scales[0, :I, 1] = 1 / 64
    gu_codes[0, I:] = 12
    gu_scales[0, I:] = 1 / 64
    d_codes = np.zeros((E, H, I), np.uint8)
    d_scales = np.zeros((E, H, I // 32), np.float16)
    d_codes[0, 0::2] = 7
    d_codes[0, 1::2] = 10
    d_scales[0] = 0.5
    return x, wr, gu_codes, gu_scales, d_codes, d_scales


def test_prefill_hand_computed_layer():
    x, wr, gc, gs, dc, ds = _hand_layer(1.0)
    out, r = O.moe_prefill(x, wr, gc, gs, dc, ds, k=1)
    assert r["idx"].tolist() == [[0]] and r["w"].tolist() == [[1.0]]
    # g = 32*1*(1/32) + 32*1*(1/64) = 1.5 ; u = 64*4*(1/64) = 4
    # h = silu(1.5) * 4 = 6 / (1 + e^-1.5)
    h = 6.0 / (1.0 + math.exp(-1.5))
    assert abs(h - 4.905446857161862) < 1e-12
    # even rows: 0.5 * (-1) * 32 h = -16 h ; odd rows: 0.5 * 2 * 32 h = 32 h ; plus x = 1
    expect = np.where(np.arange(64) % 2 == 0, 1.0 - 16 * h, 1.0 + 32 * h)
    assert np.allclose(out[0], expect, rtol=0, atol=1e-10)
    # with k = 2 the zero-scale expert adds nothing and expert 0 is weighted by
    # softmax(64 * 1/64, 0)[0] = 1 / (1 + e^-1)
    out2, r2 = O.moe_prefill(x, wr, gc, gs, dc, ds, k=2)
    w0 = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(w0 - 0.7310585786300049) < 1e-15
    assert abs(r2["w"][0, 0] - w0) < 1e-14
    expect2 = 1.0 + w0 * np.where(np.arange(64) % 2 == 0, -16 * h, 32 * h)
    assert np.allclose(out2[0], expect2, rtol=0, atol=1e-10)


def test_decode_hand_computed_layer_exact_integers():
    # x = 127 everywhere: d_x = fp16(127/127) = 1, q_x = 127.
    x, wr, gc, gs, dc, ds = _hand_layer(127.0)
    out, st = O.moe_decode(x, wr, gc, gs, dc, ds, k=1, keep_dots=True)
    assert np.all(st["qx"] == 127) and np.all(st["dx"].astype(np.float64) == 1.0)
    G = st["dots_gu"][(0, 0)]
    assert np.all(G[:32] == 32 * 127)           # gate: (9-8)*127 per element
    assert np.all(G[32:] == 4 * 32 * 127)       # up:   (12-8)*127
    # g = 4064/32 + 4064/64 = 190.5 ; u = 2 * 16256/64 = 508 ; h = silu(190.5)*508 = 96774
    assert np.all(st["h"][0, 0] == 96774.0)
    # h quantises exactly: 96774 / 127 = 762 -> d_h = 762, q_h = 127
    assert np.all(st["qh"] == 127) and np.all(st["dh"].astype(np.float64) == 762.0)
    D = st["dots_d"][(0, 0)]
    assert np.all(D[0::2] == -32 * 127) and np.all(D[1::2] == 2 * 32 * 127)
    # y = 0.5 * 762 * D ; out = 127 + y
    expect = np.where(np.arange(64) % 2 == 0, 127.0 - 1548384.0, 127.0 + 3096768.0)
    assert np.array_equal(out[0], expect)
    # the prefill evaluation of the same exactly-representable case agrees
    outp, _ = O.moe_prefill(x, wr, gc, gs, dc, ds, k=1)
    assert np.array_equal(outp[0], expect)


@pytest.mark.parametrize("evaluate", ["prefill", "decode"])
def test_zero_scales_give_identity(evaluate):
    li = workloads.tiny()
    zs = np.zeros_like(li.gu_scales)
    fn = O.moe_prefill if evaluate == "prefill" else O.moe_decode
    out, _ = fn(li.x, li.wr, li.gu_codes, zs, li.d_codes, li.d_scales, li.k)
    assert np.array_equal(out, O.bf16_bits_to_f64(li.x))
    out, _ = fn(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, np.zeros_like(li.d_scales), li.k)
    assert np.array_equal(out, O.bf16_bits_to_f64(li.x))


def test_bucketed_equals_dense_bruteforce():
    li = workloads.make_layer("small", 12, 64, 32, 5, 2, seed=11, wr_std=0.1)
    out, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    dense = O.moe_dense_bruteforce(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    assert np.allclose(out, dense, rtol=0, atol=1e-12 * max(1.0, np.abs(dense).max()))


def test_token_subset_matches_full_rows():
    li = workloads.tiny()
    full, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    sub, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k,
                           tokens=[3, 17, 40])
    assert np.allclose(sub, full[[3, 17, 40]], rtol=0, atol=1e-12)


def test_down_scale_doubling_doubles_the_moe_term():
    li = workloads.tiny()
    X = O.bf16_bits_to_f64(li.x)
    a, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    b, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes,
                         (li.d_scales.astype(np.float32) * 2).astype(np.float16), li.k)
    assert np.allclose(b - X, 2 * (a - X), rtol=0, atol=1e-12)
    # doubling the up scales doubles h, hence the MoE term, too
    gs = li.gu_scales.copy()
    gs[:, li.I:] = (gs[:, li.I:].astype(np.float32) * 2).astype(np.float16)
    c, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, gs, li.d_codes, li.d_scales, li.k)
    assert np.allclose(c - X, 2 * (a - X), rtol=0, atol=1e-12)


def test_single_expert_is_a_dense_swiglu_ffn():
    # E = 1, k = 1: routing weight 1, the layer is x + W_d (silu(W_g x) * W_u x)
    li = workloads.make_layer("one", 5, 64, 32, 1, 1, seed=12, wr_std=0.1)
    out, r = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, 1)
    assert np.all(r["w"] == 1.0)
    import torch
    X = torch.tensor(O.bf16_bits_to_f64(li.x))
    W = torch.tensor(li.gu_codes[0].astype(np.float64) - 8) * torch.tensor(
        np.repeat(li.gu_scales[0].astype(np.float64), 32, axis=-1))
    Wd = torch.tensor(li.d_codes[0].astype(np.float64) - 8) * torch.tensor(
        np.repeat(li.d_scales[0].astype(np.float64), 32, axis=-1))
    g, u = X @ W[:32].T, X @ W[32:].T
    ref = X + (torch.nn.functional.silu(g) * u) @ Wd.T
    assert np.allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_decode_close_to_prefill_on_tiny():
    li = workloads.tiny()
    a, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    b, st = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    X = O.bf16_bits_to_f64(li.x)
    # int8 activations carry ~1/254 relative error per element; the MoE term
    # should move by a small fraction of its size
    rel = O.rms(b - a) / O.rms(a - X)
    assert rel < 0.03, rel
    # stage consistency: routing identical to prefill's
    assert np.array_equal(st["idx"], O.route(X, li.wr, li.k)[1])


# ------------------------------------------------------------ stacked pre-norm
def test_rmsnorm_properties():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((6, 256)) * 3.0
    xn = O.bf16_bits_to_f64(O.rmsnorm_bf16_bits(X))
    # unit mean square up to the bf16 rounding of each element
    assert np.allclose(np.mean(xn * xn, axis=1), 1.0, atol=1e-2)
    # invariant under exact (power-of-two) scaling of the row
    for c in (0.25, 8.0, -2.0):
        xs = O.bf16_bits_to_f64(O.rmsnorm_bf16_bits(X * c))
        assert np.array_equal(xs, np.sign(c) * xn)
    # a constant row c maps to sign(c) / sqrt(1 + eps / c^2): 1 in bf16
    const = O.bf16_bits_to_f64(O.rmsnorm_bf16_bits(np.full((1, 64), -5.0)))
    assert np.all(const == -1.0)


def test_bf16_rounding_ties_to_even():
    a = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -7, -(1.0 + 2.0 ** -8)])
    assert O.f64_to_bf16_bits(a).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80]


def test_prenorm_layer_residual_and_norm():
    li = workloads.make_layer("pn", 12, 256, 128, 8, 2, seed=51, wr_std=0.05)
    args = (li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    X = O.bf16_bits_to_f64(li.x)
    # the residual is x itself, not its normalised copy
    zero = (li.wr, li.gu_codes, li.gu_scales, li.d_codes, np.zeros_like(li.d_scales), li.k)
    out0, _ = O.moe_prefill(li.x, *zero, prenorm=True)
    assert np.array_equal(out0, X)
    # the MoE term sees RMSNorm(x): scaling x by 4 scales only the residual
    x4 = O.f64_to_bf16_bits(X * 4.0)
    o1, r1 = O.moe_prefill(li.x, *args, prenorm=True)
    o4, r4 = O.moe_prefill(x4, *args, prenorm=True)
    assert np.array_equal(r1["idx"], r4["idx"])
    assert np.allclose(o4 - 4.0 * X, o1 - X, rtol=0, atol=1e-12)
    # without the norm the MoE term does change with the scale
    p1, _ = O.moe_prefill(li.x, *args)
    p4, _ = O.moe_prefill(x4, *args)
    assert not np.allclose(p4 - 4.0 * X, p1 - X, atol=1e-3)
    # decode applies the same norm before its int8 codes
    d0, _ = O.moe_decode(li.x, *zero, prenorm=True)
    assert np.array_equal(d0, X)


def test_stack_equals_layer_composition():
    layers = [workloads.make_layer("st", 9, 256, 128, 6, 2, seed=60 + l, wr_std=0.05) for l in range(2)]
    x0 = layers[0].x

    def layer(l):
        li = layers[l]
        return li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales

    xb = x0
    for l in range(2):
        out, _ = O.moe_prefill(xb, *layer(l), 2, prenorm=True)
        xb = O.f64_to_bf16_bits(out)
    assert np.array_equal(O.moe_stack_prefill(x0, layer, 2, 2), xb)
    # a subset of tokens gives the same rows (each token is independent)
    sub = O.moe_stack_prefill(x0, layer, 2, 2, tokens=[1, 7])
    assert np.array_equal(sub, xb[[1, 7]])


def test_rmsnorm_eps_inside_the_root_hand_worked():
    # A row of 2^-10 (exact in bf16): mean square 2^-20 = 9.5367431640625e-7,
    # plus eps 1e-6 gives 1.95367431640625e-6, whose root is 1.3977390e-3;
    # 2^-10 over that is 0.6987712 = 1.3975424 x 2^-1, which bf16 (7 stored
    # mantissa bits: 1.3975424 x 128 = 178.89 -> 179) rounds to 179/256 =
    # 0.69921875, bits 0x3F33.  With eps outside the root the quotient would
    # be 0.99902 (bf16 1.0, 0x3F80), and without eps exactly 1.0.
    xn = O.rmsnorm_bf16_bits(np.full((1, 64), 2.0 ** -10))
    assert np.all(xn == 0x3F33)
    # a zero row stays zero (eps keeps the root positive)
    assert np.all(O.rmsnorm_bf16_bits(np.zeros((1, 32))) == 0)


def test_stack_prefill_hand_worked_two_layers():
    # Layer 0 is the hand layer above (its router sends every token to expert
    # 0, k = 1) and its input is 2.0 everywhere.  The pre-norm gives
    # 2 / sqrt(4 + 1e-6) = 0.99999988, 1.0 in bf16, so the MoE term is the
    # hand-computed one for x = 1 (h = 6 / (1 + e^-1.5) = 4.9054469) and the
    # residual is 2: even rows 2 - 16 h = -76.487 -> bf16 -76.5, odd rows
    # 2 + 32 h = 158.97 -> bf16 159.0 (both 8 significant bits).
    # Layer 1 has all scales zero, so its MoE term vanishes and its output is
    # its residual, which must be layer 0's output (not the stack's input).
    x, wr, gc, gs, dc, ds = _hand_layer(2.0)
    zero = (wr, gc, np.zeros_like(gs), dc, np.zeros_like(ds))

    def layer(l):
        return (wr, gc, gs, dc, ds) if l == 0 else zero

    expect = O.f64_to_bf16_bits(np.where(np.arange(64) % 2 == 0, -76.5, 159.0))[None, :]
    assert np.array_equal(O.moe_stack_prefill(x, layer, 1, 1), expect)
    assert np.array_equal(O.moe_stack_prefill(x, layer, 2, 1), expect)
    # the layers are taken in order: the zero layer first leaves x unchanged
    # and the hand layer then acts on it
    swapped = lambda l: layer(1 - l)  # noqa: E731
    assert np.array_equal(O.moe_stack_prefill(x, swapped, 1, 1), x)
    assert np.array_equal(O.moe_stack_prefill(x, swapped, 2, 1), expect)
