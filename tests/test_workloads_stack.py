"""The counter-based generator of the stacked workload (CPU).

Both implementations (numpy for the oracle, torch for the GPU) must give the
same bits, and they must be SplitMix64 as published (Steele, Lea, Flood,
OOPSLA 2014): the first output of the stream seeded with 0 is the widely
quoted 0xE220A8397B1DCDAF.
"""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")


def test_splitmix64_known_answer():
    assert int(W.splitmix64_np(np.array([0], np.uint64), 0)[0]) == 0xE220A8397B1DCDAF
    t = W.splitmix64_torch(torch.tensor([0]), 0)
    assert int(t[0]) & ((1 << 64) - 1) == 0xE220A8397B1DCDAF


def test_numpy_and_torch_generators_agree():
    idx = np.array([0, 1, 2, 12345, 2 ** 40 + 7, 2 ** 62 + 3], np.uint64)
    a = W.splitmix64_np(idx, 4)
    b = W.splitmix64_torch(torch.tensor(idx.astype(np.int64)), 4).numpy().astype(np.uint64)
    assert np.array_equal(a, b)
    for layer, e in ((0, 0), (39, 255)):
        ref = W.stacked_expert(layer, e)
        got = W.stacked_experts_torch(layer, e, e + 1, "cpu")
        for r, g in zip(ref, got):
            g = g[0].numpy()
            if r.dtype == np.float16:
                assert np.array_equal(r.view(np.uint16), g.view(np.uint16))
            else:
                assert np.array_equal(r, g)


def test_stacked_expert_ranges_and_independence():
    gc, gs, dc, ds = W.stacked_expert(5, 9)
    assert gc.shape == (1536, 2048) and dc.shape == (2048, 768)
    assert gc.min() == 0 and gc.max() == 15 and abs(gc.mean() - 7.5) < 0.05
    for s in (gs, ds):
        f = s.astype(np.float32)
        assert f.min() >= 0.005 - 1e-5 and f.max() <= 0.02 + 1e-5
    # another expert or layer draws different values
    assert not np.array_equal(W.stacked_expert(5, 10)[0], gc)
    assert not np.array_equal(W.stacked_expert(6, 9)[0], gc)
    # the lazy view draws the same expert
    lz = W.stacked_layer_lazy(5)
    assert np.array_equal(lz[1][9], gc) and np.array_equal(lz[4][9].view(np.uint16), ds.view(np.uint16))
