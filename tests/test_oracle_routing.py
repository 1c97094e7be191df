"""Pins for the oracle's router top-k, bucketing and activation quantiser (CPU).

The pages ("A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011
GPU", Methodology 1 and 2) name MoE routing, a grouped GEMM over the routed
experts and 8-bit decode activations without printing formulas; the checks
here tie the oracle to exact arithmetic, brute force and library routines
that do not share its code.
"""
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

from oracle import moe_oracle as O
import workloads


def _bf16_round(a):
    return O.bf16_bits_to_f64(workloads.f32_to_bf16_bits(np.asarray(a, np.float32)))


def test_router_logits_exact_rational():
    rng = np.random.default_rng(1)
    T, H, E = 3, 40, 5
    xb = workloads.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = rng.standard_normal((E, H)).astype(np.float32)
    X = O.bf16_bits_to_f64(xb)
    L = O.router_logits(X, wr)
    assert L.shape == (T, E)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(X[t, h])) * Fraction(float(wr[e, h])) for h in range(H))
            assert abs(Fraction(float(L[t, e])) - exact) <= Fraction(1, 2**40) * (1 + abs(exact))


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(2)
    T, E, k = 50, 9, 4
    # small integers make many exact ties
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float64)
    idx = O.topk_select(logits, k)
    for t in range(T):
        ref = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert idx[t].tolist() == ref


def test_topk_duplicate_router_rows_tie_to_lower_index():
    rng = np.random.default_rng(3)
    H = 64
    wr = rng.standard_normal((6, H)).astype(np.float32)
    wr[4] = wr[1]                      # experts 1 and 4 always tie exactly
    x = workloads.f32_to_bf16_bits(rng.standard_normal((200, H)).astype(np.float32))
    L, idx, w = O.route(O.bf16_bits_to_f64(x), wr, 3)
    for t in range(200):
        sel = idx[t].tolist()
        if 4 in sel:
            assert 1 in sel and sel.index(1) < sel.index(4)


def test_topk_weights_sum_to_one_and_order():
    li = workloads.tiny()
    L, idx, w = O.route(O.bf16_bits_to_f64(li.x), li.wr, li.k)
    assert np.allclose(w.sum(-1), 1.0, atol=1e-12, rtol=0)
    sel = np.take_along_axis(L, idx, -1)
    assert np.all(np.diff(sel, axis=-1) <= 0)          # descending logits
    assert np.all(np.diff(w, axis=-1) <= 1e-15)        # hence descending weights
    # selected logits dominate every unselected one
    mask = np.ones_like(L, bool)
    np.put_along_axis(mask, idx, False, -1)
    assert np.all(sel[:, -1:] >= np.where(mask, L, -np.inf).max(-1, keepdims=True))


def test_k_equals_E_is_full_softmax():
    li = workloads.tiny()
    L, idx, w = O.route(O.bf16_bits_to_f64(li.x), li.wr, li.E)
    full = softmax(L, axis=-1)
    assert np.allclose(np.take_along_axis(full, idx, -1), w, atol=1e-14, rtol=0)


def test_bucket_bruteforce_and_invariants():
    rng = np.random.default_rng(4)
    T, E, k = 37, 7, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    off, tok, slot = O.bucket(idx, E)
    assert off[0] == 0 and off[-1] == T * k and np.all(np.diff(off) >= 0)
    for e in range(E):
        pairs = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        got = list(zip(tok[off[e]:off[e + 1]].tolist(), slot[off[e]:off[e + 1]].tolist()))
        assert got == pairs                            # ascending token order
    # every token appears in exactly k buckets, each time with a distinct slot
    for t in range(T):
        assert sorted(slot[tok == t].tolist()) == list(range(k))


def test_bucket_empty_experts():
    idx = np.array([[0, 2], [2, 0], [0, 2]])
    off, tok, slot = O.bucket(idx, 5)
    assert off.tolist() == [0, 3, 3, 6, 6, 6]
    assert tok.tolist() == [0, 1, 2, 0, 1, 2] and slot.tolist() == [0, 1, 0, 1, 0, 1]


# ---------------------------------------------------------------- act quant
def _all_fp16_positive():
    h = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)  # finite, > 0
    return h.astype(np.float64)


def _round_to_fp16_exact(fr: Fraction, table):
    """Nearest fp16 to a positive rational, ties to even, saturating at 65504."""
    import bisect
    vals, fracs = table
    if fr >= Fraction(65504):
        return 65504.0
    i = bisect.bisect_left(fracs, fr)
    if i == 0:
        lo, hi = Fraction(0), fracs[0]
        lo_bits, hi_bits = 0, 1
    else:
        lo, hi = fracs[i - 1], fracs[i] if i < len(fracs) else None
        lo_bits, hi_bits = i, i + 1
    if hi is None or fr == lo:
        return float(lo)
    if fr == hi:
        return float(hi)
    dlo, dhi = fr - lo, hi - fr
    if dlo < dhi:
        return float(lo)
    if dhi < dlo:
        return float(hi)
    return float(lo) if lo_bits % 2 == 0 else float(hi)


def test_act_scale_exhaustive_over_bf16():
    """d = fp16(fp32(amax / 127)) equals the exact rational amax/127 rounded
    to fp16 (nearest even) for every positive finite bf16 amax."""
    vals = _all_fp16_positive()
    table = (vals, [Fraction(float(v)) for v in vals])
    bits = np.arange(1, 0x7F80, dtype=np.uint16)     # all positive finite bf16
    amax = O.bf16_bits_to_f32(bits)
    g = np.zeros((bits.size, 32), np.float32)
    g[:, 0] = amax
    _, d = O.act_quant(g)
    got = d[:, 0].astype(np.float64)
    # check exactly where it matters: every value whose fp16 result is a
    # normal or subnormal number or saturates
    for i in range(0, bits.size, 1):
        a = float(amax[i])
        exact = _round_to_fp16_exact(Fraction(a) / 127, table)
        if got[i] != exact:
            raise AssertionError(f"amax={a!r}: got {got[i]!r}, exact {exact!r}")


def test_act_code_rounding_matches_exact_rational():
    """q = round-half-away(fp32(x / d)) equals the exact rational rounding for
    every positive bf16 x against a spread of fp16 scales (all exponents)."""
    xb = np.arange(1, 0x7F80, dtype=np.uint16)
    x = O.bf16_bits_to_f32(xb)
    rng = np.random.default_rng(6)
    d_bits = np.unique(np.concatenate([
        np.arange(0x0001, 0x7C00, 0x0400, dtype=np.uint16),          # one per exponent
        rng.integers(0x0001, 0x7C00, size=200).astype(np.uint16),
        np.array([0x3C00, 0x2008, 0x1C08, 0x0001, 0x7BFF], np.uint16),
    ]))
    for db in d_bits:
        d32 = np.float32(np.array([db], np.uint16).view(np.float16)[0])
        with np.errstate(over="ignore"):
            r32 = (x / d32).astype(np.float32).astype(np.float64)
        q32 = np.clip(np.sign(r32) * np.floor(np.abs(r32) + 0.5), -127, 127)
        # exact decision: n = floor(x/d + 1/2), done in float64 where the f64
        # quotient is far from a half-integer, and in rationals where it is not
        r64 = x.astype(np.float64) / np.float64(d32)
        q64 = np.clip(np.floor(r64 + 0.5), -127, 127)
        near = np.abs((r64 - np.floor(r64)) - 0.5) < 1e-9
        near &= r64 < 128
        for i in np.nonzero(near)[0]:
            fr = Fraction(float(x[i])) / Fraction(float(d32))
            n = (fr + Fraction(1, 2)).__floor__()
            q64[i] = max(-127, min(127, n))
        bad = np.nonzero(q32 != q64)[0]
        assert bad.size == 0, (float(d32), x[bad[:5]], q32[bad[:5]], q64[bad[:5]])


def test_act_quant_properties():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((50, 256)) * rng.uniform(0.01, 100, (50, 1))).astype(np.float32)
    v[3, 32:64] = 0.0                                      # a zero group
    q, d = O.act_quant(v)
    dd = np.repeat(d.astype(np.float64), 32, -1)
    assert np.all(np.abs(q) <= 127)
    assert np.all(q[3, 32:64] == 0) and d[3, 1] == 0
    # reconstruction within half a step except where the clamp bites
    err = np.abs(q * dd - v.astype(np.float64))
    clamped = np.abs(q) == 127
    assert np.all(err[~clamped] <= 0.5 * dd[~clamped] * (1 + 2**-20))
    # the largest magnitude of each group maps to +-127
    g = v.reshape(50, 8, 32)
    pos = np.abs(g).argmax(-1)
    qg = q.reshape(50, 8, 32)
    top = np.take_along_axis(qg, pos[..., None], -1)[..., 0]
    nz = d.astype(np.float64) > 0
    assert np.all(np.abs(top[nz]) == 127)
    # signs follow the input
    assert np.all(np.sign(q[q != 0]) == np.sign(v[q != 0]))


def test_act_quant_round_half_away_at_exact_halves():
    # d = 1 (amax = 127): values k + 0.5 round away from zero
    g = np.zeros((1, 32), np.float32)
    g[0, :7] = [127.0, 0.5, -0.5, 2.5, -2.5, 126.5, -1.5]
    q, d = O.act_quant(g)
    assert float(d[0, 0]) == 1.0
    assert q[0, :7].tolist() == [127, 1, -1, 3, -3, 127, -2]


def test_group_dots_second_formula():
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 16, size=(24, 128)).astype(np.uint8)
    qa = rng.integers(-127, 128, size=(3, 128))
    G = O.group_dots(codes, qa)
    # sum (q - 8) a = sum q a - 8 sum a, per block of 32, in plain Python ints
    for b in range(3):
        for r in range(24):
            for g in range(4):
                sl = slice(32 * g, 32 * g + 32)
                s_qa = int(np.dot(codes[r, sl].astype(np.int64), qa[b, sl]))
                s_a = int(qa[b, sl].sum())
                assert G[b, r, g] == s_qa - 8 * s_a
    # worst case magnitude fits int32 with room: 32 * 8 * 127
    worst = O.group_dots(np.zeros((1, 32), np.uint8), np.full(32, -127))
    assert worst[0, 0] == 32 * 8 * 127
