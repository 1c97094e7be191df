"""GPU: the 8-bit-weight decode layer (moe_w8a8_forward_decode with
weights packed by moe_q8_pack) through the C ABI, against the oracle's 8-bit
path (moe_decode with wbits=8).

The companion page "A Modern Multimodal Assistant on a 6 GB 2011 GPU:
Stage-Validated, All-GPU CUDA Inference for Fermi" (Abstract) runs 8-bit
weights against 4-bit ones at decode; the format is the Q8_0-style reading
of the oracle (blocks of 32 int8 codes, one fp16 scale, w = d * q).

Cases:
* genuine 8-bit codes over the whole range at T = 1, 4 and 16 of the decode
  shape: routing and the int8 codes of x exact, the gate/up and down int32
  group dots bit-exact (down: the oracle's dots of the GPU's own h codes), h
  codes within one step, the output within 2e-2 of the output's RMS;
* edge shapes: one token, k = E, one expert, the smallest hidden size, 16
  tokens over 64 experts (routing, gate/up dots, output);
* 12 tokens of two kinds (buckets of 6 and 12 rows, cut into slices);
* a 4-bit layer written as 8-bit codes (q - 8, same scales): the 8-bit call
  gives the 4-bit call's output bit for bit;
* the shape limit.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer, assert_within_tol, out_to_f64  # noqa: E402


def _to_q8(codes4, scales4, rng):
    # finer 8-bit codes near the 4-bit weights: q8 = 16 (q4 - 8) + noise, d8 = d4 / 16
    q = (codes4.astype(np.int32) - 8) * 16 + rng.integers(-8, 9, codes4.shape)
    q8 = np.clip(q, -127, 127).astype(np.int8)
    d8 = (scales4.astype(np.float32) / 16).astype(np.float16)
    return q8, d8


def _pack8(codes, scales):
    E, N, K = codes.shape
    c = torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scales).view(np.int16)).cuda()
    return moe.moe_q8_pack(c, s, E, N, K)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_w8_decode_against_the_oracle(T):
    li = W.decode(T)
    rng = np.random.default_rng(100 + T)
    gu8, gus8 = _to_q8(li.gu_codes, li.gu_scales, rng)
    d8, ds8 = _to_q8(li.d_codes, li.d_scales, rng)
    dl = DeviceLayer(li)
    wgu, wd = _pack8(gu8, gus8), _pack8(d8, ds8)
    d, dbg = moe.make_debug(moe.MOE_MODE_DECODE, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(moe.moe_w8a8_forward_decode(dl.x, dl.wr, wgu, wd, li.I, li.k, debug=dbg))
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    ref, st = O.moe_decode(li.x, li.wr, gu8, gus8, d8, ds8, li.k, keep_dots=True, wbits=8)
    idx = d["topk_idx"].cpu().numpy()
    assert np.array_equal(idx, st["idx"])
    assert np.array_equal(d["q_x"].cpu().numpy().astype(np.int64), st["qx"])
    tok = d["bucket_token"].cpu().numpy()
    slot = d["bucket_slot"].cpu().numpy()
    dots_gu = d["dots_gu"].cpu().numpy()
    dots_d = d["dots_d"].cpu().numpy()
    q_h = d["q_h"].cpu().numpy().astype(np.int64)
    for p in range(li.T * li.k):
        t, j = tok[p], slot[p]
        assert np.array_equal(dots_gu[p], st["dots_gu"][(t, j)]), f"gate/up dots differ at row {p}"
        assert np.array_equal(dots_d[p], O.group_dots8(d8[idx[t, j]], q_h[p])), f"down dots at row {p}"
    qh_o = np.stack([st["qh"][tok[p], slot[p]] for p in range(li.T * li.k)])
    diff = np.abs(q_h - qh_o)
    assert diff.max() <= 1 and (diff > 0).mean() < 0.01
    assert_within_tol(out, ref, tol=2e-2)


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 256, 128, 8, 2),      # one token, few experts
    (3, 256, 128, 6, 6),      # k = E
    (1, 384, 256, 1, 1),      # one expert: a dense SwiGLU FFN, 3 row blocks
    (5, 128, 128, 3, 2),      # smallest hidden size
    (16, 256, 128, 64, 4),    # 16 tokens over 64 experts
])
def test_w8_edge_shapes(T, H, I, E, k):
    li = W.make_layer("w8edge", T, H, I, E, k, seed=11 * T + H + E, wr_std=0.1)
    rng = np.random.default_rng(T + E)
    gu8, gus8 = _to_q8(li.gu_codes, li.gu_scales, rng)
    d8, ds8 = _to_q8(li.d_codes, li.d_scales, rng)
    dl = DeviceLayer(li)
    wgu, wd = _pack8(gu8, gus8), _pack8(d8, ds8)
    d, dbg = moe.make_debug(moe.MOE_MODE_DECODE, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(moe.moe_w8a8_forward_decode(dl.x, dl.wr, wgu, wd, li.I, li.k, debug=dbg))
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    ref, st = O.moe_decode(li.x, li.wr, gu8, gus8, d8, ds8, li.k, keep_dots=True, wbits=8)
    assert np.array_equal(d["topk_idx"].cpu().numpy(), st["idx"])
    tok = d["bucket_token"].cpu().numpy()
    slot = d["bucket_slot"].cpu().numpy()
    dots_gu = d["dots_gu"].cpu().numpy()
    for p in range(li.T * li.k):
        assert np.array_equal(dots_gu[p], st["dots_gu"][(tok[p], slot[p])]), f"gate/up dots at row {p}"
    assert_within_tol(out, ref, tol=2e-2)


def test_w8_concentrated_buckets():
    # 12 tokens of two kinds: buckets of 6 or 12 rows, cut into slices
    li = W.decode(16)
    li.T = 12
    li.x = li.x[np.arange(12) % 2].copy()
    rng = np.random.default_rng(7)
    gu8, gus8 = _to_q8(li.gu_codes, li.gu_scales, rng)
    d8, ds8 = _to_q8(li.d_codes, li.d_scales, rng)
    dl = DeviceLayer(li)
    wgu, wd = _pack8(gu8, gus8), _pack8(d8, ds8)
    out = out_to_f64(moe.moe_w8a8_forward_decode(dl.x, dl.wr, wgu, wd, li.I, li.k))
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    ref, _ = O.moe_decode(li.x, li.wr, gu8, gus8, d8, ds8, li.k, wbits=8)
    assert_within_tol(out, ref, tol=2e-2)


@pytest.mark.parametrize("T", [1, 16])
def test_w8_with_4bit_codes_equals_the_4bit_layer(T):
    li = W.decode(T)
    dl = DeviceLayer(li)
    gu8 = (li.gu_codes.astype(np.int16) - 8).astype(np.int8)
    d8 = (li.d_codes.astype(np.int16) - 8).astype(np.int8)
    wgu, wd = _pack8(gu8, li.gu_scales), _pack8(d8, li.d_scales)
    o4 = moe.moe_w4a8_forward_decode(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k, prenorm=True)
    o8 = moe.moe_w8a8_forward_decode(dl.x, dl.wr, wgu, wd, li.I, li.k, prenorm=True)
    torch.cuda.synchronize()
    assert torch.equal(o4.view(torch.int32), o8.view(torch.int32))


def test_w8_shape_limit():
    li = W.make_layer("w8lim", 17, 256, 128, 8, 2, seed=3, wr_std=0.1)
    dl = DeviceLayer(li)
    with pytest.raises(moe.MoeError) as ex:
        moe.moe_w8a8_forward_decode(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k)
    assert ex.value.code == moe.MOE_ERR_SHAPE
