"""Planted mistakes in the oracle (CPU only).

Each mutant replaces one oracle function with a plausible wrong version (an
off-by-one offset, swapped projections, the opposite tie order, a dropped
offset, another rounding rule, the other nibble order, the norm's eps
outside the root, stacked layers that all read the stack's input); with it in place at
least one of the listed pins must fail.  This shows the pins can tell the
oracle's definitions from their likely misreadings.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
import test_oracle_golden as PG
import test_oracle_layer as PL
import test_oracle_q4 as PQ
import test_oracle_routing as PR


def dequant_offset7(codes, scales):
    codes = np.asarray(codes)
    *lead, K = codes.shape
    q = codes.astype(np.int64) - 7
    d = np.asarray(scales).astype(np.float64)
    return (q.reshape(*lead, K // O.GROUP, O.GROUP) * d[..., None]).reshape(*lead, K)


def split_up_gate(gu, I):
    return gu[..., I:, :], gu[..., :I, :]


def topk_ties_to_higher_index(logits, k):
    T, E = logits.shape
    index_key = np.broadcast_to(np.arange(E), logits.shape)
    order = np.lexsort((-index_key, -logits), axis=-1)
    return order[:, :k].astype(np.int64)


def group_dots_no_offset(codes, qa):
    w = np.asarray(codes).astype(np.int64)
    a = np.asarray(qa).astype(np.int64)
    R, K = w.shape
    prod = a[..., None, :] * w
    return prod.reshape(*prod.shape[:-1], K // O.GROUP, O.GROUP).sum(axis=-1)


def act_quant_half_even(v32):
    v32 = np.asarray(v32, dtype=np.float32)
    *lead, K = v32.shape
    g = v32.reshape(*lead, K // O.GROUP, O.GROUP)
    amax = np.abs(g).max(axis=-1)
    d16 = np.minimum((amax / np.float32(127.0)).astype(np.float32),
                     np.float32(O.FP16_MAX)).astype(np.float16)
    d32 = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (g / np.where(d32 != 0, d32, np.float32(1))).astype(np.float32).astype(np.float64)
    q = np.where(d32 != 0, np.clip(np.rint(r), -127, 127), 0).astype(np.int64)
    return q.reshape(*lead, K), d16


def blocks18_nibbles_swapped(blocks):
    blocks = np.asarray(blocks, dtype=np.uint8)
    *lead, nb, _ = blocks.shape
    scales = np.ascontiguousarray(blocks[..., 0:2]).view("<f2")[..., 0].astype(np.float16)
    qs = blocks[..., 2:18]
    codes = np.concatenate([qs >> 4, qs & 0x0F], axis=-1)
    return codes.reshape(*lead, nb * O.GROUP), scales


def rmsnorm_eps_outside_root(X):
    X = np.asarray(X, dtype=np.float64)
    r = 1.0 / (np.sqrt(np.mean(X * X, axis=-1, keepdims=True)) + O.RMS_EPS)
    return O.f64_to_bf16_bits(X * r)


def stack_every_layer_reads_the_input(x_bits, layer, L, k, tokens=None, keep=False):
    xb = np.asarray(x_bits)
    out = xb
    for l in range(L):
        wr, gc, gs, dc, ds = layer(l)
        o, _ = O.moe_prefill(xb, wr, gc, gs, dc, ds, k, prenorm=True)
        out = O.f64_to_bf16_bits(o)
    return out


MUTANTS = {
    "offset -7": ("q4_dequant", dequant_offset7,
                  [PQ.test_dequant_worked_example_two_blocks, PG.test_q4_0_blocks18_decode,
                   PL.test_prefill_hand_computed_layer]),
    "gate and up swapped": ("_split_gate_up", split_up_gate,
                            [PL.test_prefill_hand_computed_layer,
                             PL.test_decode_hand_computed_layer_exact_integers]),
    "ties to the higher index": ("topk_select", topk_ties_to_higher_index,
                                 [PR.test_topk_bruteforce_with_ties,
                                  PR.test_topk_duplicate_router_rows_tie_to_lower_index,
                                  PG.test_router_topk_cases]),
    "group dots without the -8": ("group_dots", group_dots_no_offset,
                                  [PG.test_w4a8_group_dot, PR.test_group_dots_second_formula,
                                   PL.test_decode_hand_computed_layer_exact_integers]),
    "codes rounded half to even": ("act_quant", act_quant_half_even,
                                   [PR.test_act_quant_round_half_away_at_exact_halves,
                                    PG.test_w4a8_group_dot]),
    "eps outside the root": ("rmsnorm_bf16_bits", rmsnorm_eps_outside_root,
                             [PL.test_rmsnorm_eps_inside_the_root_hand_worked]),
    "stacked layers all read the input": ("moe_stack_prefill", stack_every_layer_reads_the_input,
                                          [PL.test_stack_prefill_hand_worked_two_layers]),
    "nibble order swapped": ("q4_from_blocks18", blocks18_nibbles_swapped,
                             [PQ.test_blocks18_hand_built, PG.test_q4_0_blocks18_decode]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    attr, mutant, pins = MUTANTS[name]
    for pin in pins:  # the pins pass on the oracle as it is
        pin()
    monkeypatch.setattr(O, attr, mutant)
    failed = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
