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
* skewed   T=10240, same shapes, expert popularity a water-filled Zipf(1.1)
           law through a calibrated bias channel, 16 experts never chosen,
           seed 3
* stacked  a 40-layer stack of pre-norm layers, T=4096, H=2048, I=768, E=256,
           k=8, fresh weights per layer (27.2 GB packed), seed 4.  Its
           weights come from a counter-based generator (below) so that the
           GPU can draw all of them and the oracle only the experts a sampled
           token reaches, bit for bit the same.

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


def zipf_water_filled(n: int, k: int, s: float) -> np.ndarray:
    """Per-rank selection fractions f_r = min(1, c * r^-s), r = 1..n, with c
    chosen (bisection) so that sum_r f_r = k: a Zipf law of exponent s
    water-filled under the cap of 1 (an expert cannot be chosen by more than
    every token)."""
    base = np.arange(1, n + 1, dtype=np.float64) ** -s
    lo, hi = 0.0, float(k) * n / base.sum()
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(1.0, c * base).sum() > k:
            hi = c
        else:
            lo = c
    return np.minimum(1.0, 0.5 * (lo + hi) * base)


def _gaussian_selection_prob(b: np.ndarray, sig: np.ndarray, k: int, z: np.ndarray) -> np.ndarray:
    """P_i = Pr(fewer than k of the other variables exceed L_i) for independent
    L_i ~ N(b_i, sig_i^2): the density of L_i integrated (on the uniform grid
    z) against the Poisson-binomial probability that at most k - 1 of the
    others lie above it.  The count distribution of the others is built from
    prefix and suffix products over the variables, truncated at k."""
    from scipy.special import ndtr
    n, G = b.size, z.size
    p = ndtr((b[:, None] - z[None, :]) / sig[:, None])        # Pr(L_j > z)

    def step(q, pj):
        nxt = q * (1.0 - pj)[:, None]
        nxt[:, 1:] += q[:, :-1] * pj[:, None]
        nxt[:, k] += q[:, k] * pj                              # state k means ">= k"
        return nxt

    pre = np.zeros((n + 1, G, k + 1))
    pre[0, :, 0] = 1.0
    for j in range(n):
        pre[j + 1] = step(pre[j], p[j])
    suf = np.zeros((n + 1, G, k + 1))
    suf[n, :, 0] = 1.0
    for j in range(n - 1, -1, -1):
        suf[j] = step(suf[j + 1], p[j])
    below = np.cumsum(suf[1:, :, :k], axis=2)                 # Pr(suffix count <= m)
    q = np.einsum("igm,igm->ig", pre[:-1, :, :k], below[:, :, ::-1])
    dens = np.exp(-0.5 * ((z[None, :] - b[:, None]) / sig[:, None]) ** 2) / (
        sig[:, None] * np.sqrt(2.0 * np.pi))
    return (dens * q).sum(axis=1) * (z[1] - z[0])


def calibrate_zipf_biases(sig: np.ndarray, k: int, s: float, T: int) -> np.ndarray:
    """Biases b (one per live expert, in rank order) such that, with logits
    b_i + N(0, sig_i^2) drawn independently per token, expert i is among a
    token's k largest with probability f_i of ``zipf_water_filled``.  An
    expert whose f_i is capped at 1 is pushed up until it misses fewer than
    half a token in T.  Deterministic fixed-point iterations: b_i moves by
    half the log ratio of target to current probability (the logit ratio for
    capped experts, which only move up), re-centred on the uncapped mean
    (the probabilities do not change under a common shift)."""
    n = sig.size
    f = zipf_water_filled(n, k, s)
    cap = f >= 1.0
    target = np.where(cap, 1.0 - 0.5 / T, f)

    def logit(v):
        return np.log(v) - np.log1p(-v)

    b = np.log(f)
    for _ in range(400):
        z = np.linspace(b.min() - 8.0 * sig.max(), b.max() + 8.0 * sig.max(), 600)
        P = np.clip(_gaussian_selection_prob(b, sig, k, z), 1e-12, 1.0 - 1e-12)
        d = np.where(cap, np.maximum(0.0, logit(target) - logit(P)), np.log(target) - np.log(P))
        if np.abs(d).max() < 1e-4:
            break
        b += np.clip(0.5 * d, -0.5, 0.5)
        b -= b[~cap].mean()
    return b


_SKEWED_CACHE: dict = {}


def skewed(seed: int = 3, T: int = 10240, zipf_s: float = 1.1, dead: int = 16) -> LayerInputs:
    """Long prefill whose expert popularity follows a water-filled Zipf law.

    The last hidden channel is a constant 1 (a bias channel), so the router's
    weight on it, b_e, is added to expert e's logit exactly.  Experts are
    ranked by a seeded permutation; the last ``dead`` of them get b = -1e4 and
    are never chosen.  For the E - dead live ones, b is calibrated so that the
    fraction of tokens choosing the expert of rank r is f_r = min(1, c r^-s)
    with sum_r f_r = k (``zipf_water_filled``; at s = 1.1 the rank-1 expert is
    chosen by every token, rank 80 by ~1.7% and rank 112 by ~1.2%).  The
    calibration treats the rest of each logit, x[:, :H-1] . wr[e, :H-1], as
    independent N(0, |wr[e, :H-1]|^2) noise (x ~ N(0, 1)) and solves for b by
    fixed-point iterations on the Gaussian order statistics
    (``calibrate_zipf_biases``); the realised histogram of the actual tokens
    then follows the targets up to sampling noise.  The other router weights
    are N(0, 0.02).
    """
    key = (seed, T, zipf_s, dead)
    if key not in _SKEWED_CACHE:
        H, I, E, k = 2048, 768, 128, 8
        li = make_layer("skewed", T, H, I, E, k, seed, 0.02)
        rng = np.random.Generator(np.random.PCG64(seed + 1000))
        perm = rng.permutation(E)
        live = perm[: E - dead]
        sig = np.sqrt(np.sum(li.wr[live, : H - 1].astype(np.float64) ** 2, axis=1))
        b_live = calibrate_zipf_biases(sig, k, zipf_s, T)
        bias = np.full(E, -1.0e4, dtype=np.float64)
        bias[live] = b_live
        li.wr[:, H - 1] = bias.astype(np.float32)
        li.x[:, H - 1] = f32_to_bf16_bits(np.ones(1, np.float32))[0]
        li.notes = {"zipf_s": zipf_s, "dead_experts": sorted(int(e) for e in perm[E - dead:]),
                    "rank_order": [int(e) for e in live],
                    "target_fraction": zipf_water_filled(E - dead, k, zipf_s).tolist()}
        _SKEWED_CACHE[key] = li
    src = _SKEWED_CACHE[key]
    return dataclasses.replace(src, x=src.x.copy(), wr=src.wr.copy(), gu_codes=src.gu_codes,
                               gu_scales=src.gu_scales, d_codes=src.d_codes,
                               d_scales=src.d_scales, notes=dict(src.notes))


# --------------------------------------------------------------------------
# Counter-based weights for the stacked workload
# --------------------------------------------------------------------------
# SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
# generators", OOPSLA 2014): output i of the stream with seed s is
# mix(s + (i + 1) * GAMMA), mix(z) = z1 ^ (z1 >> 31) with
# z1 = (z0 ^ (z0 >> 27)) * M2, z0 = (z ^ (z >> 30)) * M1, all modulo 2^64.
# The index of a value encodes (layer, expert, part, row, block):
#   i = (((layer * 512 + expert) * 4 + part) * 4096 + row) * 256 + block
# part 0: gate/up codes, 1: down codes (one output = 16 codes, code c of the
# block in bits 4c..4c+3), 2: gate/up scales, 3: down scales (one output per
# 32-column group: d = fp16(fp32(0.005 + 0.015 * (out >> 11) / 2^53))).
STACK = dict(L=40, T=4096, H=2048, I=768, E=256, k=8, seed=4)
SM_GAMMA = 0x9E3779B97F4A7C15
SM_M1 = 0xBF58476D1CE4E5B9
SM_M2 = 0x94D049BB133111EB
_U64 = (1 << 64) - 1


def _stack_index(layer, expert, part, row, block):
    return (((layer * 512 + expert) * 4 + part) * 4096 + row) * 256 + block


def splitmix64_np(index: np.ndarray, seed: int) -> np.ndarray:
    """SplitMix64 outputs for uint64 stream positions ``index`` (numpy)."""
    z = np.asarray(index, dtype=np.uint64) + np.uint64(1)
    z = z * np.uint64(SM_GAMMA) + np.uint64(seed & _U64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(SM_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(SM_M2)
    return z ^ (z >> np.uint64(31))


def splitmix64_torch(index, seed: int):
    """The same outputs for an int64 torch tensor of positions (two's
    complement int64 arithmetic; right shifts masked to act as logical)."""
    import torch

    def c64(v):  # unsigned 64-bit constant as a signed int64
        v &= _U64
        return v - (1 << 64) if v >= 1 << 63 else v

    def lsr(z, n):
        return (z >> n) & ((1 << (64 - n)) - 1)

    z = (index.to(torch.int64) + 1) * c64(SM_GAMMA) + c64(seed)
    z = (z ^ lsr(z, 30)) * c64(SM_M1)
    z = (z ^ lsr(z, 27)) * c64(SM_M2)
    return z ^ lsr(z, 31)


def _codes_from_words_np(words: np.ndarray) -> np.ndarray:
    shifts = (np.arange(16, dtype=np.uint64) * np.uint64(4))
    return ((words[..., None] >> shifts) & np.uint64(15)).astype(np.uint8).reshape(*words.shape[:-1], -1)


def _scales_from_words_np(words: np.ndarray) -> np.ndarray:
    # fp64 -> fp32 -> fp16, the same two roundings on both generators
    u = (words >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return (0.005 + 0.015 * u).astype(np.float32).astype(np.float16)


def stacked_expert(layer: int, expert: int, seed: int = STACK["seed"], H: int = STACK["H"],
                   I: int = STACK["I"]):
    """One expert of one stacked layer on the host: (gu_codes [2I, H],
    gu_scales [2I, H/32], d_codes [H, I], d_scales [H, I/32])."""
    def words(part, rows, cols_per_word, ncols):
        r = np.arange(rows, dtype=np.uint64)[:, None]
        b = np.arange(ncols // cols_per_word, dtype=np.uint64)[None, :]
        idx = (((np.uint64(layer) * np.uint64(512) + np.uint64(expert)) * np.uint64(4) +
                np.uint64(part)) * np.uint64(4096) + r) * np.uint64(256) + b
        return splitmix64_np(idx, seed)
    gu_codes = _codes_from_words_np(words(0, 2 * I, 16, H))
    d_codes = _codes_from_words_np(words(1, H, 16, I))
    gu_scales = _scales_from_words_np(words(2, 2 * I, GROUP, H))
    d_scales = _scales_from_words_np(words(3, H, GROUP, I))
    return gu_codes, gu_scales, d_codes, d_scales


def stacked_experts_torch(layer: int, e0: int, e1: int, device, seed: int = STACK["seed"],
                          H: int = STACK["H"], I: int = STACK["I"]):
    """Experts e0..e1-1 of one stacked layer as torch tensors on ``device``:
    codes uint8 [n, 2I, H] / [n, H, I] and scales float16, equal bit for bit
    to ``stacked_expert``."""
    import torch
    n = e1 - e0
    e = torch.arange(e0, e1, device=device, dtype=torch.int64)[:, None, None]

    def words(part, rows, cols_per_word, ncols):
        r = torch.arange(rows, device=device, dtype=torch.int64)[None, :, None]
        b = torch.arange(ncols // cols_per_word, device=device, dtype=torch.int64)[None, None, :]
        idx = (((layer * 512 + e) * 4 + part) * 4096 + r) * 256 + b
        return splitmix64_torch(idx, seed)

    def codes(w):
        sh = torch.arange(16, device=device, dtype=torch.int64) * 4
        c = ((w[..., None] >> sh) & 15).to(torch.uint8)  # low bits only: the sign fill is masked
        return c.reshape(n, w.shape[1], -1)

    def scales(w):
        u = ((w >> 11) & ((1 << 53) - 1)).to(torch.float64) * 2.0 ** -53
        return (0.005 + 0.015 * u).to(torch.float32).to(torch.float16)

    return codes(words(0, 2 * I, 16, H)), scales(words(2, 2 * I, GROUP, H)), \
        codes(words(1, H, 16, I)), scales(words(3, H, GROUP, I))


def stacked_router(layer: int, seed: int = STACK["seed"]) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed * 1000 + layer))
    return (rng.standard_normal((STACK["E"], STACK["H"]), dtype=np.float32) *
            np.float32(0.02)).astype(np.float32)


def stacked_x(seed: int = STACK["seed"], T: int = STACK["T"]) -> np.ndarray:
    return _hidden(np.random.Generator(np.random.PCG64(seed)), T, STACK["H"])


class LazyExperts:
    """Array-like view of one stacked layer's experts for the oracle: indexing
    by expert draws (and caches) that expert from the counter-based stream."""

    def __init__(self, layer: int, which: int, seed: int = STACK["seed"]):
        self.layer, self.which, self.seed = layer, which, seed
        H, I, E = STACK["H"], STACK["I"], STACK["E"]
        self.shape = [(E, 2 * I, H), (E, 2 * I, H // GROUP), (E, H, I), (E, H, I // GROUP)][which]
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            self._cache[e] = stacked_expert(self.layer, e, self.seed)
        return self._cache[e][self.which]


def stacked_layer_lazy(layer: int, seed: int = STACK["seed"]):
    """(wr, gu_codes, gu_scales, d_codes, d_scales) of a stacked layer, the
    weights as LazyExperts (sharing one per-expert cache)."""
    gc = LazyExperts(layer, 0, seed)
    views = [gc] + [LazyExperts(layer, w, seed) for w in (1, 2, 3)]
    for v in views[1:]:
        v._cache = gc._cache
    return (stacked_router(layer, seed), *views)


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
