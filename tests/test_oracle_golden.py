"""The oracle against the hand-worked fixtures in tests/golden/ (CPU only).

Each fixture states its source passage and works its expected values by
hand from the definitions there (Q4_0 block decoding, the W4A8 group dot,
router top-k order and weights); the oracle must reproduce them exactly, or
to within double-precision rounding where an exponential is involved.
"""
import os

import numpy as np

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _records(name):
    """(key, value) pairs of a fixture, comments and blank lines skipped."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, _, val = line.partition(":")
                out.append((key.strip(), val.strip()))
    return out


def test_q4_0_blocks18_decode():
    recs = _records("q4_0_blocks18.txt")
    blocks = [bytes.fromhex(v) for k, v in recs if k == "block"]
    weights = [[float(t) for t in v.split()] for k, v in recs if k == "weights"]
    assert len(blocks) == len(weights) == 2
    for raw, want in zip(blocks, weights):
        assert len(raw) == 18 and len(want) == 32
        codes, scales = O.q4_from_blocks18(np.frombuffer(raw, dtype=np.uint8)[None, :])
        assert O.q4_dequant(codes, scales).tolist() == want


def test_w4a8_group_dot():
    r = dict(_records("w4a8_group_dot.txt"))
    v = np.array([float(t) for t in r["c"].split()], dtype=np.float32) / np.float32(16)
    q, d = O.act_quant(v)
    assert float(d[0]) == float(r["scale_a"])
    assert q.tolist() == [int(t) for t in r["q"].split()]
    codes = np.array([[int(t) for t in r["codes"].split()]], dtype=np.uint8)
    assert O.group_dots(codes, q).tolist() == [[int(r["dot"])]]
    y, _ = O.w4a8_rows(codes, np.array([[float(r["scale_w"])]], dtype=np.float16), q, d)
    assert y.tolist() == [float(r["y"])]


def test_router_topk_cases():
    cases = [v for k, v in _records("router_topk.txt") if k == "case"]
    assert len(cases) == 3
    for c in cases:
        k, logits, picked, weights = (part.split() for part in c.split("|"))
        lg = np.array([[float(t) for t in logits]])
        idx = O.topk_select(lg, int(k[0]))
        assert idx.tolist() == [[int(t) for t in picked]]
        w = O.topk_weights(lg, idx)
        np.testing.assert_allclose(w[0], [float(t) for t in weights], rtol=1e-14, atol=0)
