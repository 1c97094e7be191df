"""GPU parity of whole layers against the oracle, through the C ABI.

Float outputs: max|gpu - oracle| <= 2e-2 * RMS(oracle output) per layer (in the
fp32 output mode; the bf16 mode adds half a bf16 ulp of the oracle value).
Integer stages of the W4A8 decode path are bit-exact: the int8 activation
codes and scales, the int32 gate/up group dots, and the int32 down group dots
recomputed by the oracle from the GPU's own int8 codes of h (h itself is fp32
on the GPU and float64 in the oracle, so a code of h may differ by one at a
rounding boundary; such differences are counted and bounded).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer, assert_within_tol, out_to_f64  # noqa: E402


def _sample_tokens(T, n, seed=0):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    s.update({0, T - 1})
    return np.array(sorted(s))


# ------------------------------------------------------------------ prefill
def test_prefill_tiny_full():
    li = workloads.tiny()
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_PREFILL, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(dl.prefill(debug=dbg))
    ref, r = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    assert np.array_equal(d["topk_idx"].cpu().numpy(), r["idx"])
    assert_within_tol(out, ref)
    # a stricter view: the MoE term alone (out - x) is within 1% too
    X = O.bf16_bits_to_f64(li.x)
    assert_within_tol(out - X, ref - X, tol=1e-2, what="MoE term")
    # stage: h = silu(W_g x) * (W_u x) per bucket row, fp16
    h = d["h"].cpu().numpy().astype(np.float64)
    tok = d["bucket_token"].cpu().numpy()
    off = d["expert_offsets"].cpu().numpy()
    href = np.zeros_like(h)
    for e in range(li.E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        W = O.q4_dequant(li.gu_codes[e], li.gu_scales[e])
        Xe = X[tok[rows]]
        href[rows] = O.swiglu(Xe @ W[: li.I].T, Xe @ W[li.I:].T)
    assert_within_tol(h, href, tol=1e-2, what="h")


def test_prefill_tiny_bf16_output():
    li = workloads.tiny()
    out = out_to_f64(DeviceLayer(li).prefill(out_fp32=False))
    ref, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    half_ulp = np.abs(ref) * 2.0 ** -8
    r = O.rms(ref)
    assert np.all(np.abs(out - ref) <= 2e-2 * r + half_ulp)


@pytest.mark.parametrize("name,nsample", [("prefill", 48), ("skewed", 24)])
def test_prefill_full_size_sampled(name, nsample):
    li = workloads.CONFIGS[name]()
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_PREFILL, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(dl.prefill(debug=dbg))
    toks = _sample_tokens(li.T, nsample, seed=3)
    ref, r = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k,
                           tokens=toks)
    assert_within_tol(out[toks], ref)
    # stage: the sampled tokens' rows of h = silu(W_g x) * (W_u x), fp16, in
    # bucket order, each against the oracle's for the expert of its bucket
    h = d["h"].cpu().numpy()
    tok = d["bucket_token"].cpu().numpy()
    slot = d["bucket_slot"].cpu().numpy()
    X = O.bf16_bits_to_f64(li.x)
    got, want = [], []
    for i, t in enumerate(toks):
        for p in np.nonzero(tok == t)[0]:
            e = r["idx"][i, slot[p]]
            W = O.q4_dequant(li.gu_codes[e], li.gu_scales[e])
            want.append(O.swiglu(W[: li.I] @ X[t], W[li.I:] @ X[t]))
            got.append(h[p].astype(np.float64))
    assert len(got) == len(toks) * li.k
    assert_within_tol(np.array(got), np.array(want), tol=1e-2, what="h (sampled rows)")
    # every row is finite and the residual dominates nowhere unexpectedly
    assert np.all(np.isfinite(out))
    # deterministic: a second call gives the same bits
    out2 = out_to_f64(dl.prefill())
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 256, 128, 8, 2),      # a single token
    (37, 256, 128, 8, 2),     # ragged token count
    (300, 256, 128, 2, 1),    # buckets larger than one 256-token tile
    (40, 256, 128, 6, 6),     # k = E: every token uses every expert
    (9, 384, 256, 1, 1),      # one expert: a dense SwiGLU FFN; 3 row blocks
    (700, 128, 128, 3, 2),    # smallest hidden size, several tiles per expert
])
def test_prefill_edge_shapes(T, H, I, E, k):
    li = workloads.make_layer("edge", T, H, I, E, k, seed=T + H + E, wr_std=0.1)
    out = out_to_f64(DeviceLayer(li).prefill())
    ref, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, k)
    assert_within_tol(out, ref)


def test_prefill_zero_scales_identity_and_empty():
    li = workloads.tiny()
    li.d_scales[:] = 0
    dl = DeviceLayer(li)
    out = out_to_f64(dl.prefill())
    assert np.array_equal(out, O.bf16_bits_to_f64(li.x))
    # T = 0 is a no-op
    x0 = torch.empty((0, li.H), dtype=torch.bfloat16, device="cuda")
    o0 = moe.moe_q4_forward_prefill(x0, dl.wr, dl.wgu, dl.wd, li.I, li.k)
    assert o0.shape == (0, li.H)


# ------------------------------------------------------------------- decode
def _decode_check(li, tol=2e-2):
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_DECODE, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(dl.decode(debug=dbg))
    ref, st = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k,
                           keep_dots=True)
    idx = d["topk_idx"].cpu().numpy()
    assert np.array_equal(idx, st["idx"]), "routing differs from the oracle"
    # bucket membership and order: bit-exact against the oracle's bucketing
    off_o, tok_o, slot_o = O.bucket(st["idx"], li.E)
    assert np.array_equal(d["expert_offsets"].cpu().numpy(), off_o)
    assert np.array_equal(d["bucket_token"].cpu().numpy(), tok_o)
    assert np.array_equal(d["bucket_slot"].cpu().numpy(), slot_o)
    # int8 activations and their scales: bit-exact
    assert np.array_equal(d["q_x"].cpu().numpy().astype(np.int64), st["qx"])
    assert np.array_equal(d["d_x"].cpu().numpy().view(np.uint16), st["dx"].view(np.uint16))
    # gate/up int32 group dots: bit-exact, bucket order
    tok = d["bucket_token"].cpu().numpy()
    slot = d["bucket_slot"].cpu().numpy()
    dots_gu = d["dots_gu"].cpu().numpy()
    dots_d = d["dots_d"].cpu().numpy()
    q_h = d["q_h"].cpu().numpy().astype(np.int64)
    for p in range(li.T * li.k):
        t, j = tok[p], slot[p]
        assert np.array_equal(dots_gu[p], st["dots_gu"][(t, j)]), f"gate/up dots differ at row {p}"
        # down dots: the oracle's integer dots of the GPU's own q_h
        e = idx[t, j]
        assert np.array_equal(dots_d[p], O.group_dots(li.d_codes[e], q_h[p])), f"down dots at row {p}"
    # q_h vs the oracle's: within one code
    qh_o = np.stack([st["qh"][tok[p], slot[p]] for p in range(li.T * li.k)])
    diff = np.abs(q_h - qh_o)
    assert diff.max() <= 1
    assert (diff > 0).mean() < 0.01
    assert_within_tol(out, ref, tol=tol)
    return out


@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_full_size(T):
    _decode_check(workloads.decode(T))


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 256, 128, 8, 2),      # one token, few experts (all-thread top-k path)
    (2, 256, 128, 8, 2),      # two tokens (one-warp bucketing)
    (2, 2048, 768, 128, 8),   # two tokens at full size
    (3, 256, 128, 6, 6),      # k = E
    (1, 384, 256, 1, 1),      # one expert: a dense SwiGLU FFN, 3 row blocks
    (5, 128, 128, 3, 2),      # smallest hidden size
    (16, 256, 128, 64, 4),    # more (token, expert) logits than threads of a CTA, E < 128
    (32, 256, 128, 32, 2),    # the same on the task kernel (T > 16)
])
def test_decode_edge_shapes(T, H, I, E, k):
    _decode_check(workloads.make_layer("dedge", T, H, I, E, k, seed=7 * T + H + E, wr_std=0.1))


@pytest.mark.parametrize("T,groups", [
    (16, 1),   # all 16 tokens alike: 8 buckets of 16 rows, eight slices each
    (12, 2),   # two kinds of token: buckets of 6 (three slices) or 12 (six)
    (9, 3),    # buckets of 3, 6 or 9 rows (slices of 1 and 2 rows)
    (5, 1),    # buckets of 5: slices of 1, 2 and 2 rows
    (4, 2),    # T <= 4: buckets of 2 or 4 rows, a slice per row
])
def test_decode_concentrated_buckets(T, groups):
    # tokens repeated so that many choose the same experts: the clustered
    # kernel cuts each bucket into slices of at most two rows (one for T <= 4)
    li = workloads.decode(16)
    rows = np.arange(T) % groups
    li.T = T
    li.x = li.x[rows].copy()
    _decode_check(li)


def test_decode_tiny_32_tokens():
    li = workloads.tiny()
    li.T = 32
    li.x = li.x[:32].copy()
    _decode_check(li)


def test_decode_adversarial_integer_extremes():
    # activations all +127 (q_x = 127); gate codes 15 (q - 8 = 7), up codes 0
    # (q - 8 = -8): group dots of 32*7*127 and -32*8*127, the largest there
    # are.  h is then about -6e8, so its fp16 scale saturates at 65504 and
    # every code of h clamps to -127; the down codes 15 give 32*7*(-127).
    li = workloads.make_layer("extreme", 3, 256, 128, 4, 2, seed=41, wr_std=0.1)
    li.gu_codes[:, : li.I] = 15
    li.gu_codes[:, li.I:] = 0
    li.d_codes[:] = 15
    li.x[:] = workloads.f32_to_bf16_bits(np.full(256, 127.0, np.float32))[None, :]
    _decode_check(li)


def test_decode_bf16_output():
    li = workloads.decode(4)
    dl = DeviceLayer(li)
    out = out_to_f64(dl.decode(out_fp32=False))
    ref, _ = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    half_ulp = np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(out - ref) <= 2e-2 * O.rms(ref) + half_ulp)
    # the bf16 output is the fp32 output rounded once
    out32 = dl.decode(out_fp32=True)
    assert np.array_equal(out, out_to_f64(out32.to(torch.bfloat16)))


@pytest.mark.parametrize("T", [1, 4])
def test_decode_prenorm(T):
    # MOE_STACKED_PRENORM: route and multiply RMSNorm(x), add x itself.  The
    # norm is taken in fp32 on the GPU and in float64 by the oracle, so an
    # element of the normalised x can differ by one bf16 ulp and its int8
    # code by one; the routing follows the contract, the output the layer
    # tolerance.
    li = workloads.decode(T)
    X = O.bf16_bits_to_f64(li.x)
    li.x = O.f64_to_bf16_bits(X * 7.0 + 3.0)  # an input whose norm is not ~1
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_DECODE, li.T, li.H, li.I, li.E, li.k)
    out = out_to_f64(moe.moe_w4a8_forward_decode(dl.x, dl.wr, dl.wgu, dl.wd, li.I, li.k,
                                                  debug=dbg, prenorm=True))
    ref, st = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales,
                           li.k, prenorm=True)
    assert np.array_equal(d["topk_idx"].cpu().numpy(), st["idx"])
    qx = d["q_x"].cpu().numpy().astype(np.int64)
    assert np.abs(qx - st["qx"]).max() <= 1 and (qx != st["qx"]).mean() < 0.01
    assert_within_tol(out, ref)
    # without the flag the same call gives a different layer
    plain = out_to_f64(dl.decode())
    assert not np.allclose(plain, out, atol=1e-3)


def test_decode_deterministic():
    # every sum runs in a fixed order: repeated calls give the same bits
    for T in (1, 16):
        dl = DeviceLayer(workloads.decode(T))
        a = out_to_f64(dl.decode())
        for _ in range(3):
            assert np.array_equal(out_to_f64(dl.decode()), a)


def test_shared_workspace_decode_prefill_decode():
    # One buffer serves a decode call, then a prefill call, then a decode call
    # again on the same stream: nothing a call reads may depend on what an
    # earlier call of the other path left in the buffer.
    li = workloads.decode(16)
    dl = DeviceLayer(li)
    ref_d, _ = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    ref_p, _ = O.moe_prefill(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    nb = max(moe.moe_workspace_bytes(m, li.T, li.H, li.I, li.E, li.k)
             for m in (moe.MOE_MODE_PREFILL, moe.MOE_MODE_DECODE))
    ws = torch.full((nb,), 0x7F, dtype=torch.uint8, device="cuda")
    outs = [dl.decode(workspace=ws), dl.prefill(workspace=ws), dl.decode(workspace=ws),
            dl.prefill(workspace=ws), dl.decode(workspace=ws)]
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    for i, o in enumerate(outs):
        assert_within_tol(out_to_f64(o), ref_p if i % 2 else ref_d)
    assert np.array_equal(out_to_f64(outs[0]), out_to_f64(outs[4]))


def test_decode_matches_prefill_closely():
    li = workloads.decode(16)
    dl = DeviceLayer(li)
    a = out_to_f64(dl.decode())
    b = out_to_f64(dl.prefill())
    X = O.bf16_bits_to_f64(li.x)
    assert O.rms(a - b) < 0.05 * O.rms(b - X)


def test_decode_workspace_garbage_and_reuse():
    # Every call clears the counters its kernels synchronise on: a workspace
    # full of garbage, alternating workspaces and the default allocation all
    # give the oracle's layer.
    li = workloads.decode(1)
    dl = DeviceLayer(li)
    ref, _ = O.moe_decode(li.x, li.wr, li.gu_codes, li.gu_scales, li.d_codes, li.d_scales, li.k)
    nbytes = moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, li.T, li.H, li.I, li.E, li.k)
    ws_a = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    ws_b = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    for ws in (ws_a, ws_a, ws_b, ws_b, ws_a, None, None, ws_b):
        out = out_to_f64(dl.decode(workspace=ws))
        torch.cuda.synchronize()
        assert moe.moe_get_device_status() == 0
        assert_within_tol(out, ref)
        if ws is not None:
            ws.fill_(0x3C)  # garbage again before the next use


@pytest.mark.parametrize("path", ["prefill", "decode"])
def test_layer_while_another_stream_holds_an_sm(path):
    # The expert kernels of both paths have CTAs that wait on one another, so
    # they are launched cooperatively: they start only once every CTA can be
    # resident.  A kernel on another stream that holds one SM for ~2.5 s
    # (longer than the kernels' 2 s bound on any wait) delays the layer
    # instead of making it time out.
    li = workloads.prefill() if path == "prefill" else workloads.decode(16)
    dl = DeviceLayer(li)
    ref = out_to_f64(dl.prefill() if path == "prefill" else dl.decode())
    torch.cuda.synchronize()
    other = torch.cuda.Stream()
    with torch.cuda.stream(other):
        torch.cuda._sleep(int(2.5 * 2.07e9))  # cycles: >= 2.5 s at the 2.07 GHz maximum clock
    out = out_to_f64(dl.prefill() if path == "prefill" else dl.decode())
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    assert np.array_equal(out, ref)
