"""Seeded synthetic inputs for the 4-bit MoE expert-FFN layer.

This module is shared by the CPU oracle (``oracle/``), the tests and ``bench.py``.
It draws random numbers and lays them out; it holds none of the layer's
arithmetic (no dequantisation, routing, quantisation or FFN math).

Every array is produced by ``numpy.random.Generator(PCG64(seed))`` so both sides
of a parity test see the same bits.  Layouts (all row-major, contiguous):

* ``x``         uint16 [T, H]        bf16 bit patterns of the hidden states
* ``wr``        float32 [E, H]       router weights
* ``gu_codes``  uint8 [E, 2I, H]     4-bit codes 0..15 of the gate (rows 0..I-1)
                                     and up (rows I..2I-1) projections
* ``gu_scales`` float16 [E, 2I, H/32] one scale per 32 consecutive codes
* ``d_codes``   uint8 [E, H, I]      down projection codes
* ``d_scales``  float16 [E, H, I/32]

A weight is w = d * (q - 8) (Q4_0 family); that decoding lives in the oracle and
in the kernels, not here.

Workload recipes (the page "A 35B Hybrid-Attention Mixture-of-Experts Model on a
6GB 2011 GPU", Methodology: a Q4_0-family MoE with 128 experts after pruning,
top-8 routing; the shapes follow that model family):

* tiny     T=64,  H=256,  I=128, E=8,   k=2, x~N(0,1), wr~N(0,0.05), seed 0
* decode   T in {1,4,16}, H=2048, I=768, E=128, k=8, wr~N(0,1/sqrt(H)) so the
           router logits are ~N(0,1), seed 1
* prefill  T=2048, H=2048, I=768, E=128, k=8, wr~N(0,0.02), seed 2
* skewed   T=10240, same shapes, Zipf(1.1) expert popularity through a bias
           channel, 16 experts never chosen, seed 3
* stacked  one layer of a 40-layer stack, T=4096, H=2048, I=768, E=256, k=8,
           fresh weights per layer, seed 4

Codes are uniform on 0..15; scales are uniform on [0.005, 0.02] rounded to fp16.
"""
from __future__ import annotations

import dataclasses

import numpy as np

GROUP = 32


@dataclasses.dataclass
class LayerInputs:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    seed: int
    x: np.ndarray          # uint16 [T, H] bf16 bits
    wr: np.ndarray         # float32 [E, H]
    gu_codes: np.ndarray   # uint8 [E, 2I, H]
    gu_scales: np.ndarray  # float16 [E, 2I, H/32]
    d_codes: np.ndarray    # uint8 [E, H, I]
    d_scales: np.ndarray   # float16 [E, H, I/32]
    notes: dict = dataclasses.field(default_factory=dict)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform 4-bit codes: both nibbles of random bytes."""
    n = int(np.prod(shape))
    raw = np.frombuffer(rng.bytes((n + 1) // 2), dtype=np.uint8)
    out = np.empty(2 * raw.size, dtype=np.uint8)
    out[0::2] = raw & 0x0F
    out[1::2] = raw >> 4
    return out[:n].reshape(shape)


def _scales(rng: np.random.Generator, shape, lo=0.005, hi=0.02) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


def _hidden(rng: np.random.Generator, T: int, H: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def make_layer(name: str, T: int, H: int, I: int, E: int, k: int, seed: int,
               wr_std: float, scale_range=(0.005, 0.02)) -> LayerInputs:
    """Draw one layer: hidden states, router, then gate/up and down experts."""
    if H % GROUP or I % GROUP:
        raise ValueError("H and I must be multiples of 32")
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _hidden(rng, T, H)
    wr = (rng.standard_normal((E, H), dtype=np.float32) * np.float32(wr_std)).astype(np.float32)
    gu_codes = _codes(rng, (E, 2 * I, H))
    gu_scales = _scales(rng, (E, 2 * I, H // GROUP), *scale_range)
    d_codes = _codes(rng, (E, H, I))
    d_scales = _scales(rng, (E, H, I // GROUP), *scale_range)
    return LayerInputs(name, T, H, I, E, k, seed, x, wr, gu_codes, gu_scales, d_codes, d_scales)


def tiny(seed: int = 0) -> LayerInputs:
    return make_layer("tiny", 64, 256, 128, 8, 2, seed, 0.05)


def decode(T: int = 1, seed: int = 1) -> LayerInputs:
    if T not in (1, 4, 16):
        raise ValueError("the decode workload is defined for T in {1, 4, 16}")
    H = 2048
    return make_layer(f"decode_T{T}", T, H, 768, 128, 8, seed, 1.0 / np.sqrt(H))


def prefill(seed: int = 2) -> LayerInputs:
    return make_layer("prefill", 2048, 2048, 768, 128, 8, seed, 0.02)


def skewed(seed: int = 3, T: int = 10240, zipf_s: float = 1.1, dead: int = 16) -> LayerInputs:
    """Long prefill whose expert popularity follows a Zipf law.

    The last hidden channel is a constant 1 (a bias channel) and the router's
    weight on it is b_e = s * ln(1 / rank_e) for the E - ``dead`` live experts
    (ranks drawn as a random permutation) and -1e4 for ``dead`` experts, which
    are then never chosen.  The other router weights are N(0, 0.02), so each
    logit carries N(0, ~0.9) noise on top of its bias; with that noise the
    chance of an expert being picked falls with its rank roughly as a Zipf law
    of exponent s (exactly so for Gumbel noise of unit scale).  The realised
    expert histogram is whatever the routing makes of these inputs.
    """
    H, I, E, k = 2048, 768, 128, 8
    li = make_layer("skewed", T, H, I, E, k, seed, 0.02)
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    perm = rng.permutation(E)
    live = perm[: E - dead]
    bias = np.full(E, -1.0e4, dtype=np.float64)
    ranks = np.arange(1, E - dead + 1, dtype=np.float64)
    bias[live] = zipf_s * np.log(1.0 / ranks)
    li.wr[:, H - 1] = bias.astype(np.float32)
    li.x[:, H - 1] = f32_to_bf16_bits(np.ones(1, np.float32))[0]
    li.notes = {"zipf_s": zipf_s, "dead_experts": sorted(int(e) for e in perm[E - dead:]),
                "rank_order": [int(e) for e in live]}
    return li


def stacked_layer(layer: int, seed: int = 4, T: int = 4096) -> LayerInputs:
    """Layer ``layer`` (0-based) of the 40-layer stack: fresh weights per layer.

    Only layer 0 carries its own hidden states; deeper layers take the previous
    layer's output.  The router is N(0, 0.02) as in the single-layer prefill.
    """
    return make_layer(f"stacked_L{layer}", T, 2048, 768, 256, 8, seed * 1000 + layer, 0.02)


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "prefill": prefill,
    "skewed": skewed,
}


def blocks18(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Lay codes/scales out as 18-byte Q4_0 blocks: fp16 scale (little-endian),
    then 16 bytes whose byte j holds element j (low nibble) and j+16 (high)."""
    *lead, K = codes.shape
    nb = K // GROUP
    c = codes.reshape(*lead, nb, GROUP)
    out = np.empty((*lead, nb, 18), dtype=np.uint8)
    out[..., 0:2] = np.ascontiguousarray(scales.astype("<f2")).view(np.uint8).reshape(*lead, nb, 2)
    out[..., 2:18] = (c[..., :16] & 0x0F) | ((c[..., 16:] & 0x0F) << 4)
    return out
