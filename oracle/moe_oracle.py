"""CPU oracle for the 4-bit (Q4_0 family) mixture-of-experts expert-FFN layer.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline leg and its
reference arm, and by nothing else.  The CUDA library never imports, links or
falls back to it; it shares no code, table or constant with the kernels.

It is a plain, slow, obviously correct restatement of what the layer computes,
in float64 for real-valued arithmetic and int64 for integer dot products.
numpy matmul and sort serve as library steps; nothing is blocked, fused or
reordered beyond the definitions below.

Source: "A 35B Hybrid-Attention Mixture-of-Experts Model on a 6GB 2011 GPU:
Hand-Written 4-bit CUDA Inference for Fermi" (gist.science, paper 2606.24031).
  * Methodology, section 1 "Hybrid GPU-Prefill / CPU-Decode": prefill runs a
    grouped 4-bit GEMM over the routed experts with floating-point
    activations; decode runs a W4A8 (4-bit weights, 8-bit activations)
    integer multiply-add kernel.
  * Methodology, section 2 "Memory and Quantization": weights use group-wise
    symmetric 4-bit quantisation of the Q4_0 family; decode activations are
    8-bit.
  * Key Contributions 2: the integer decode path.
The pages name the method but print no formula; the readings taken where they
are silent (block layout, router, activation, quantiser rounding, tie rule)
are stated beside each function and collected in the design notes.

Pins (checked in ``tests/test_oracle_*.py`` against facts that do not come from
this file): hand-worked Q4_0 encode/decode blocks; a hand-built 18-byte block;
a hand-computed one-expert layer; brute-force dense evaluation (every token
through every expert) against the bucketed one; k = E reducing to a full
softmax; exact rational checks of every quantiser rounding decision over all
bf16 magnitudes; a second, independent formula for the integer group dots;
invariants (weights sum to 1, each token in exactly k buckets, zero scales
give out = x).
"""
from __future__ import annotations

import numpy as np

GROUP = 32  # Q4_0 block: 32 consecutive weights share one fp16 scale


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly: a bf16 is the top half of an fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest, ties to even) through fp32: fp64 -> fp32 -> bf16.
    (The two roundings differ from one exact rounding only when the fp32 value
    falls exactly on a bf16 midpoint.)"""
    u = np.asarray(a, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


# --------------------------------------------------------------------------
# Pre-norm for stacked layers (reading: the pages print no layer norm; a
# stack of residual MoE layers needs one to stay finite, and the plainest is
# an RMSNorm of the layer input with unit gain)
# --------------------------------------------------------------------------
RMS_EPS = 1e-6


def rmsnorm_bf16_bits(X: np.ndarray) -> np.ndarray:
    """Per row: X / sqrt(mean(X^2) + 1e-6), rounded to bf16 bit patterns."""
    X = np.asarray(X, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(X * X, axis=-1, keepdims=True) + RMS_EPS)
    return f64_to_bf16_bits(X * r)


# --------------------------------------------------------------------------
# Q4_0-family weights (Methodology 2, "Quantization")
# --------------------------------------------------------------------------
def q4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode Q4_0 weights: w = d * (q - 8).

    ``codes`` uint8 [..., K] with values 0..15; ``scales`` fp16 [..., K/32].
    Element i of a row belongs to block i // 32, whose scale is d.  The
    product of an fp16 scale and a small integer is exact in float64.
    """
    codes = np.asarray(codes)
    *lead, K = codes.shape
    q = codes.astype(np.int64) - 8
    d = np.asarray(scales).astype(np.float64)
    return (q.reshape(*lead, K // GROUP, GROUP) * d[..., None]).reshape(*lead, K)


def q4_encode(w: np.ndarray):
    """Encode float weights into Q4_0 blocks (READING of the Q4_0 family rule).

    Per block of 32: m is the element of largest magnitude (the first one on a
    tie), sign kept; d = fp16(m / -8); q_i = min(15, floor(x_i / d + 8.5)),
    taken against the stored (fp16-rounded) d; a block of zeros has d = 0 and
    all q = 8.  d may be negative.  Returns (codes uint8, scales fp16).
    """
    w = np.asarray(w, dtype=np.float64)
    *lead, K = w.shape
    b = w.reshape(*lead, K // GROUP, GROUP)
    pos = np.argmax(np.abs(b), axis=-1)                      # first maximum
    m = np.take_along_axis(b, pos[..., None], axis=-1)[..., 0]
    d16 = (m / -8.0).astype(np.float16)
    d = d16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.floor(np.where(d != 0, b / np.where(d != 0, d, 1.0), 0.0) + 8.5)
    q = np.clip(q, 0, 15).astype(np.uint8)
    return q.reshape(*lead, K), d16


def q4_from_blocks18(blocks: np.ndarray):
    """Split 18-byte Q4_0 blocks into (codes, scales).

    Block layout (READING of the usual Q4_0 byte order): bytes 0-1 are the
    fp16 scale, little-endian; in bytes 2..17, byte j holds element j in its
    low nibble and element j + 16 in its high nibble.
    ``blocks`` uint8 [..., nb, 18] -> codes uint8 [..., nb*32], scales fp16 [..., nb].
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    *lead, nb, _ = blocks.shape
    scales = np.ascontiguousarray(blocks[..., 0:2]).view("<f2")[..., 0].astype(np.float16)
    qs = blocks[..., 2:18]
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    return codes.reshape(*lead, nb * GROUP), scales


def q8_encode(w: np.ndarray):
    """Encode float weights into 8-bit blocks (READING of a Q8_0-style rule).

    The companion page "A Modern Multimodal Assistant on a 6 GB 2011 GPU:
    Stage-Validated, All-GPU CUDA Inference for Fermi" (Abstract) runs 8-bit
    weights against 4-bit ones without printing the format; the plainest member of the
    same family: per block of 32, d = fp16(amax / 127), amax the block's
    largest magnitude; q_i = clamp(round_half_away_from_zero(x_i / d), -127,
    127), taken against the stored (fp16-rounded) d; a block of zeros has
    d = 0 and all q = 0.  Returns (codes int8, scales fp16)."""
    w = np.asarray(w, dtype=np.float64)
    *lead, K = w.shape
    b = w.reshape(*lead, K // GROUP, GROUP)
    amax = np.abs(b).max(axis=-1)
    d16 = (amax / 127.0).astype(np.float16)
    d = d16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d != 0, b / np.where(d != 0, d, 1.0), 0.0)
    q = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)
    return q.reshape(*lead, K), d16


def q8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode 8-bit weights: w = d * q (exact in float64)."""
    codes = np.asarray(codes)
    *lead, K = codes.shape
    q = codes.astype(np.int64)
    d = np.asarray(scales).astype(np.float64)
    return (q.reshape(*lead, K // GROUP, GROUP) * d[..., None]).reshape(*lead, K)


# --------------------------------------------------------------------------
# Router (Methodology 1: tokens are routed to experts before the grouped GEMM)
# --------------------------------------------------------------------------
def router_logits(x: np.ndarray, wr: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * wr[e, h] in float64.

    x is bf16 (8 significant bits) and wr fp32 (24), so every product is exact
    in float64; only the summation rounds.
    """
    return np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T


def topk_select(logits: np.ndarray, k: int) -> np.ndarray:
    """The k experts with the largest logits, in descending logit order; equal
    logits go to the lower expert index first (READING: ties are decided by
    the integer index, never by floating point)."""
    T, E = logits.shape
    index_key = np.broadcast_to(np.arange(E), logits.shape)
    order = np.lexsort((index_key, -logits), axis=-1)  # primary: -logit, then index
    return order[:, :k].astype(np.int64)


def topk_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Softmax over the k selected logits.

    This equals a softmax over all E experts renormalised over the selected k,
    since the common denominator cancels."""
    sel = np.take_along_axis(logits, idx, axis=-1)
    z = np.exp(sel - sel.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def route(x: np.ndarray, wr: np.ndarray, k: int):
    """Router top-k: returns (logits [T,E], idx [T,k], weights [T,k])."""
    logits = router_logits(x, wr)
    idx = topk_select(logits, k)
    return logits, idx, topk_weights(logits, idx)


# --------------------------------------------------------------------------
# Bucketing: the "grouped" in grouped GEMM (Methodology 1, prefill)
# --------------------------------------------------------------------------
def bucket(idx: np.ndarray, E: int):
    """Group the (token, slot) pairs by expert.

    count_e = #{(t, j) : idx[t, j] = e}; offsets is its exclusive prefix sum
    (length E + 1); bucket e lists its tokens in ascending token order, with
    the slot j at which the token chose e.  Returns (offsets, bucket_token,
    bucket_slot) as int64 arrays.
    """
    idx = np.asarray(idx)
    tok, slot = [], []
    counts = np.zeros(E, dtype=np.int64)
    for e in range(E):
        t_e, j_e = np.nonzero(idx == e)   # row-major: ascending t
        counts[e] = t_e.size
        tok.append(t_e)
        slot.append(j_e)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return offsets, np.concatenate(tok).astype(np.int64), np.concatenate(slot).astype(np.int64)


# --------------------------------------------------------------------------
# SwiGLU between gate/up and down
# --------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(gate) * up."""
    return silu(g) * u


# --------------------------------------------------------------------------
# 8-bit activations for decode (Methodology 2; Key Contributions 2)
# --------------------------------------------------------------------------
FP16_MAX = 65504.0


def act_quant(v32: np.ndarray):
    """Symmetric int8 quantisation per 32 consecutive values (READING).

    d = fp16(amax / 127), amax the group's largest magnitude, the quotient
    taken in fp32 and then rounded to fp16 (nearest even), saturating at
    65504; q = clamp(round_half_away_from_zero(v / d), -127, 127), the
    quotient taken in fp32 (the precision the kernels decide in); d = 0 gives
    q = 0.  ``v32`` float32 [..., K] -> (q int64 [..., K], d fp16 [..., K/32]).
    """
    v32 = np.asarray(v32, dtype=np.float32)
    *lead, K = v32.shape
    g = v32.reshape(*lead, K // GROUP, GROUP)
    amax = np.abs(g).max(axis=-1)
    quot = (amax / np.float32(127.0)).astype(np.float32)
    d16 = np.minimum(quot, np.float32(FP16_MAX)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (g / np.where(d32 != 0, d32, np.float32(1))).astype(np.float32).astype(np.float64)
    q = np.sign(r) * np.floor(np.abs(r) + 0.5)           # half away from zero, exact in f64
    q = np.where(d32 != 0, np.clip(q, -127, 127), 0).astype(np.int64)
    return q.reshape(*lead, K), d16


def group_dots(codes: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """W4A8 integer group dot products.

    G[..., r, g] = sum over i in block g of (codes[r, i] - 8) * qa[..., i],
    exact in int64.  ``codes`` uint8 [R, K]; ``qa`` int [..., K].
    Returns int64 [..., R, K/32].
    """
    w = np.asarray(codes).astype(np.int64) - 8
    a = np.asarray(qa).astype(np.int64)
    R, K = w.shape
    prod = a[..., None, :] * w                       # [..., R, K]
    return prod.reshape(*prod.shape[:-1], K // GROUP, GROUP).sum(axis=-1)


def w4a8_rows(codes: np.ndarray, scales: np.ndarray, qa: np.ndarray, da: np.ndarray):
    """Rows of a W4A8 projection: y_r = sum_g d_w[r, g] * d_a[g] * G[r, g].

    Returns (y float64 [..., R], G int64 [..., R, K/32])."""
    G = group_dots(codes, qa)
    dw = np.asarray(scales).astype(np.float64)
    dA = np.asarray(da).astype(np.float64)[..., None, :]
    return (dw * dA * G).sum(axis=-1), G


def group_dots8(codes: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """W8A8 integer group dot products: G[..., r, g] = sum over i in block g
    of codes[r, i] * qa[..., i], exact in int64.  ``codes`` int8 [R, K]."""
    w = np.asarray(codes).astype(np.int64)
    a = np.asarray(qa).astype(np.int64)
    R, K = w.shape
    prod = a[..., None, :] * w
    return prod.reshape(*prod.shape[:-1], K // GROUP, GROUP).sum(axis=-1)


def w8a8_rows(codes: np.ndarray, scales: np.ndarray, qa: np.ndarray, da: np.ndarray):
    """Rows of a W8A8 projection: y_r = sum_g d_w[r, g] * d_a[g] * G[r, g]."""
    G = group_dots8(codes, qa)
    dw = np.asarray(scales).astype(np.float64)
    dA = np.asarray(da).astype(np.float64)[..., None, :]
    return (dw * dA * G).sum(axis=-1), G


# --------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------
def _split_gate_up(gu: np.ndarray, I: int):
    return gu[..., :I, :], gu[..., I:, :]


def moe_prefill(x_bits, wr, gu_codes, gu_scales, d_codes, d_scales, k, tokens=None,
                prenorm=False):
    """Prefill layer with bf16 activations, computed exactly in float64.

    out[t] = x[t] + sum_j w[t, j] * W_d,e (silu(W_g,e x[t]) * (W_u,e x[t])),
    e = idx[t, j], each W the Q4_0-decoded matrix.  ``tokens`` restricts the
    evaluation to a subset of rows (routing is per token, so a row's result
    does not depend on the others).  With ``prenorm`` the router and the
    experts read xn = bf16(RMSNorm(x)) while the residual stays x.  Returns
    (out [n, H], routing dict).
    """
    X = bf16_bits_to_f64(x_bits)
    if tokens is not None:
        X = X[np.asarray(tokens)]
    residual = X
    if prenorm:
        X = bf16_bits_to_f64(rmsnorm_bf16_bits(X))
    I = gu_codes.shape[1] // 2
    logits, idx, w = route(X, wr, k)
    out = residual.copy()
    for e in np.unique(idx):
        rows, js = np.nonzero(idx == e)
        Wg, Wu = _split_gate_up(q4_dequant(gu_codes[e], gu_scales[e]), I)
        Wd = q4_dequant(d_codes[e], d_scales[e])
        Xe = X[rows]
        h = swiglu(Xe @ Wg.T, Xe @ Wu.T)
        y = h @ Wd.T
        out[rows] += w[rows, js][:, None] * y
    return out, {"logits": logits, "idx": idx, "w": w}


def moe_dense_bruteforce(x_bits, wr, gu_codes, gu_scales, d_codes, d_scales, k):
    """Every token through every expert, weighted by its routing weight (zero
    for experts it did not choose).  Slow; for tiny inputs only.  Shares the
    definitions above but none of the gather/scatter of ``moe_prefill``."""
    X = bf16_bits_to_f64(x_bits)
    T, H = X.shape
    E = gu_codes.shape[0]
    I = gu_codes.shape[1] // 2
    logits, idx, w = route(X, wr, k)
    weight = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            weight[t, idx[t, j]] = w[t, j]
    out = X.copy()
    for e in range(E):
        Wg, Wu = _split_gate_up(q4_dequant(gu_codes[e], gu_scales[e]), I)
        Wd = q4_dequant(d_codes[e], d_scales[e])
        for t in range(T):
            out[t] += weight[t, e] * (Wd @ swiglu(Wg @ X[t], Wu @ X[t]))
    return out


def moe_decode(x_bits, wr, gu_codes, gu_scales, d_codes, d_scales, k, tokens=None,
               keep_dots=False, prenorm=False, wbits=4):
    """Decode layer with W4A8 arithmetic (Methodology 1, "Decode (CPU)"), or
    with 8-bit weights (``wbits=8``: int8 codes, ``w8a8_rows``; the companion
    page's 8-bit setting) and otherwise the same steps.

    The bf16 hidden state is quantised to int8 per 32 (``act_quant``); gate
    and up rows are exact integer group dots scaled by d_w * d_x; h =
    silu(g) * u is quantised the same way (after rounding h to fp32, the
    precision in which the kernels take that decision); the down projection
    is again integer group dots, scaled by d_w * d_h and by the routing
    weight; the residual is added.  Returns (out float64 [n, H], stages)."""
    x_bits = np.asarray(x_bits)
    if tokens is not None:
        x_bits = x_bits[np.asarray(tokens)]
    residual = bf16_bits_to_f64(x_bits)
    if prenorm:
        x_bits = rmsnorm_bf16_bits(residual)
    X64 = bf16_bits_to_f64(x_bits)
    X32 = bf16_bits_to_f32(x_bits)
    n, H = X64.shape
    I = gu_codes.shape[1] // 2
    logits, idx, w = route(X64, wr, k)
    rows = w8a8_rows if wbits == 8 else w4a8_rows
    qx, dx = act_quant(X32)
    out = residual.copy()
    qh = np.zeros((n, k, I), np.int64)
    dh = np.zeros((n, k, I // GROUP), np.float16)
    hh = np.zeros((n, k, I))
    dots_gu = {} if keep_dots else None
    dots_d = {} if keep_dots else None
    for t in range(n):
        for j in range(k):
            e = idx[t, j]
            gu, G_gu = rows(gu_codes[e], gu_scales[e], qx[t], dx[t])
            h = swiglu(gu[:I], gu[I:])
            hh[t, j] = h
            qh[t, j], dh[t, j] = act_quant(h.astype(np.float32))
            y, G_d = rows(d_codes[e], d_scales[e], qh[t, j], dh[t, j])
            out[t] += w[t, j] * y
            if keep_dots:
                dots_gu[(t, j)] = G_gu
                dots_d[(t, j)] = G_d
    stages = {"logits": logits, "idx": idx, "w": w, "qx": qx, "dx": dx,
              "h": hh, "qh": qh, "dh": dh, "dots_gu": dots_gu, "dots_d": dots_d}
    return out, stages


def moe_stack_prefill(x_bits, layer, L, k, tokens=None, keep=False):
    """L stacked pre-norm prefill layers with bf16 outputs:
    x_{l+1} = bf16(x_l + MoE_l(bf16(RMSNorm(x_l)))).  ``layer(l)`` returns
    (wr, gu_codes, gu_scales, d_codes, d_scales) of layer l.  Returns the
    final bf16 bits [n, H] (and, with ``keep``, every layer's output bits and
    routing)."""
    xb = np.asarray(x_bits)
    if tokens is not None:
        xb = xb[np.asarray(tokens)]
    hist = []
    for l in range(L):
        wr, gc, gs, dc, ds = layer(l)
        out, r = moe_prefill(xb, wr, gc, gs, dc, ds, k, prenorm=True)
        xb = f64_to_bf16_bits(out)
        if keep:
            hist.append((xb, r))
    return (xb, hist) if keep else xb


def rms(a: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a)))
