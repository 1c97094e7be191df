"""The long skewed-prefill workload (CPU): expert popularity must follow a
Zipf law of exponent 1.1 water-filled under the cap of 1, as the workload
states (T=10240, E=128 with 16 experts never chosen, top-8, seed 3).

The seeded tokens are routed through the oracle and the realised tokens per
expert are compared with the targets T * min(1, c r^-1.1) (sum over ranks =
k): within binomial sampling noise at every rank, the dead experts at 0, the
rank-1 expert chosen by every token, the fitted log-log slope near -1.1.  The
histogram itself is stored in tests/golden/skewed_expert_histogram.txt
(written by make_skewed_histogram.py from the oracle) and must be reproduced
exactly.
"""
import os

import numpy as np
import pytest

import workloads as W
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "skewed_expert_histogram.txt")


def test_water_filled_zipf_targets_closed_form():
    f = W.zipf_water_filled(112, 8, 1.1)
    assert abs(f.sum() - 8.0) < 1e-9
    assert f[0] == 1.0 and np.all(f[1:] < 1.0)
    # below the cap the law is exactly c r^-1.1
    r = np.arange(1, 113, dtype=np.float64)
    c = f[1:] * r[1:] ** 1.1
    assert np.ptp(c) < 1e-12 * c[0]
    # with one capped rank: c = (k - 1) / sum_{r>=2} r^-1.1
    assert abs(c[0] - 7.0 / np.sum(r[1:] ** -1.1)) < 1e-12
    assert abs(10240 * f[79] - 172.63) < 0.01 and abs(10240 * f[111] - 119.23) < 0.01
    # no cap needed: a plain normalised Zipf law
    g = W.zipf_water_filled(1000, 2, 1.1)
    assert abs(g[0] / g[9] - 10 ** 1.1) < 1e-9 and abs(g.sum() - 2) < 1e-9


def _golden():
    rows = []
    with open(GOLDEN) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            rank, e, n, tgt = (s.strip() for s in line.split("|"))
            rows.append((int(rank), int(e), int(n), float(tgt)))
    return rows


@pytest.fixture(scope="module")
def realised():
    li = W.skewed()
    _, idx, _ = O.route(O.bf16_bits_to_f64(li.x), li.wr, li.k)
    return li, np.bincount(idx.ravel(), minlength=li.E)


def test_skewed_histogram_follows_zipf(realised):
    li, counts = realised
    order = np.asarray(li.notes["rank_order"])
    dead = np.asarray(li.notes["dead_experts"])
    assert len(order) == 112 and len(dead) == 16
    assert counts.sum() == li.T * li.k
    assert np.all(counts[dead] == 0)
    c = counts[order]
    f = np.asarray(li.notes["target_fraction"])
    assert c[0] == li.T  # capped at 1: every token
    mu = li.T * f[1:]
    sd = np.sqrt(mu * (1.0 - f[1:]))
    z = (c[1:] - mu) / sd
    assert np.max(np.abs(z)) < 4.0, f"rank {np.argmax(np.abs(z)) + 2}: z = {z.max():.2f}"
    r = np.arange(2, 113)
    slope = np.polyfit(np.log(r), np.log(c[1:]), 1)[0]
    assert abs(slope + 1.1) < 0.06, slope


def test_skewed_histogram_matches_stored(realised):
    li, counts = realised
    rows = _golden()
    assert len(rows) == li.E
    for rank, e, n, tgt in rows:
        assert counts[e] == n, f"expert {e}: {counts[e]} tokens, stored {n}"
        if rank:
            assert li.notes["rank_order"][rank - 1] == e
            assert abs(li.T * li.notes["target_fraction"][rank - 1] - tgt) < 0.01
