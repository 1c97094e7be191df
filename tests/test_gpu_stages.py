"""GPU parity of the individual stages: packing, router top-k, bucketing.

All calls go through the C ABI (ctypes binding).  Integer and index results
are compared bit for bit with the oracle; router logits are fp32 on the GPU
and float64 in the oracle, so the selection is checked by two clauses:
  1. tokens whose logit gaps (between adjacent chosen logits and between the
     k-th and (k+1)-th) exceed twice the largest observed logit error must pick
     exactly the oracle's experts in the oracle's order;
  2. every token's choice must equal the oracle's selection rule applied to the
     GPU's own fp32 logits (ties: lower expert index first), and the weights
     must be the softmax of those logits.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from gpu_util import DeviceLayer  # noqa: E402


def unpack_host(packed: np.ndarray, E: int, N: int, K: int):
    """Reads the packed layout described in include/moeq4.h back into codes
    [E,N,K] and fp16 scales [E,N,K/32]."""
    RB, KB = N // 128, K // 64
    t = packed[: E * RB * KB * 4608].reshape(E, RB, KB, 4608)
    words = np.ascontiguousarray(t[..., :4096]).view("<u4").reshape(E, RB, KB, 128, 8)
    nib = np.stack([(words >> (4 * i)) & 0xF for i in range(8)], axis=-1)  # [..., 8 words, 8 nibbles]
    cols = np.empty_like(nib)
    cols[..., 0::2] = nib[..., 0:4]   # even columns in nibbles 0..3
    cols[..., 1::2] = nib[..., 4:8]   # odd columns in nibbles 4..7
    codes = cols.reshape(E, RB, KB, 128, 64).transpose(0, 1, 3, 2, 4).reshape(E, N, K)
    sc = np.ascontiguousarray(t[..., 4096:]).view("<f2").reshape(E, RB, KB, 128, 2)
    scales = sc.transpose(0, 1, 3, 2, 4).reshape(E, N, K // 32)
    return codes.astype(np.uint8), scales


@pytest.mark.parametrize("fmt", ["codes", "blocks18"])
def test_pack_roundtrip_bit_exact(fmt):
    li = workloads.tiny()
    f = moe.MOE_Q4_CODES if fmt == "codes" else moe.MOE_Q4_BLOCK18
    dl = DeviceLayer(li, fmt=f)
    for packed, codes, scales in ((dl.wgu, li.gu_codes, li.gu_scales), (dl.wd, li.d_codes, li.d_scales)):
        E, N, K = codes.shape
        assert packed.numel() == moe.moe_q4_packed_bytes(E, N, K) == E * N * K * 18 // 32
        c, s = unpack_host(packed.cpu().numpy(), E, N, K)
        assert np.array_equal(c, codes)
        assert np.array_equal(s.view(np.uint16), scales.view(np.uint16))


def test_pack_full_size_formats_agree():
    li = workloads.make_layer("packcheck", 1, 2048, 768, 4, 1, seed=21, wr_std=0.02)
    a = DeviceLayer(li, fmt=moe.MOE_Q4_CODES)
    b = DeviceLayer(li, fmt=moe.MOE_Q4_BLOCK18)
    assert torch.equal(a.wgu, b.wgu) and torch.equal(a.wd, b.wd)
    c, s = unpack_host(a.wgu.cpu().numpy(), 4, 1536, 2048)
    assert np.array_equal(c, li.gu_codes)
    assert np.array_equal(s.view(np.uint16), li.gu_scales.view(np.uint16))


def check_routing(li, logits, idx, w):
    """Two-clause routing contract (module docstring).  Returns the number of
    near-tie tokens that only clause 2 covers."""
    X = O.bf16_bits_to_f64(li.x)
    L = O.router_logits(X, li.wr)
    lg = logits.astype(np.float64)
    delta = float(np.max(np.abs(lg - L)))
    scale = float(np.max(np.abs(L))) + 1.0
    assert delta <= 1e-4 * scale, f"router logit error {delta}"
    # clause 2: the selection rule on the GPU's own logits
    idx2 = O.topk_select(lg, li.k)
    assert np.array_equal(idx.astype(np.int64), idx2)
    assert np.allclose(w, O.topk_weights(lg, idx2), rtol=0, atol=2e-6)
    assert np.allclose(w.sum(-1), 1.0, atol=1e-5)
    # clause 1: tokens whose exact choice no logit error of the measured size
    # can change match the exact selection.  With err_e = |gpu_e - exact_e|,
    # the order of a above b is certain when L_a - L_b > err_a + err_b.
    err = np.abs(lg - L)
    idx_o = O.topk_select(L, li.k)
    clear = np.ones(len(L), bool)
    for t in range(len(L)):
        sel = idx_o[t]
        lo, hi = L[t, sel] - err[t, sel], L[t, sel] + err[t, sel]
        if li.k > 1 and np.any(lo[:-1] <= hi[1:]):
            clear[t] = False
            continue
        rest = np.ones(li.E, bool)
        rest[sel] = False
        if rest.any() and lo[-1] <= np.max(L[t, rest] + err[t, rest]):
            clear[t] = False
    assert np.array_equal(idx[clear], idx_o[clear])
    return int((~clear).sum())


def _route(dl):
    logits = torch.empty((dl.T, dl.E), dtype=torch.float32, device="cuda")
    idx, w = moe.moe_route_topk(dl.x, dl.wr, dl.k, logits=logits)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "prefill", "skewed"])
def test_route_topk(name):
    li = workloads.CONFIGS[name]()
    dl = DeviceLayer(li)
    lg, idx, w = _route(dl)
    near = check_routing(li, lg, idx, w)
    assert near <= max(2, li.T // 50), f"{near} near-tie tokens"
    # without a logits buffer the result is identical
    idx_b, w_b = moe.moe_route_topk(dl.x, dl.wr, dl.k)
    assert np.array_equal(idx_b.cpu().numpy(), idx) and np.array_equal(w_b.cpu().numpy(), w)


def test_route_exact_ties_go_to_lower_index():
    li = workloads.make_layer("ties", 300, 256, 128, 16, 4, seed=31, wr_std=0.05)
    li.wr[9] = li.wr[2]
    li.wr[15] = li.wr[2]
    dl = DeviceLayer(li)
    lg, idx, w = _route(dl)
    check_routing(li, lg, idx, w)
    for t in range(li.T):
        s = idx[t].tolist()
        for hi in (9, 15):
            if hi in s:
                assert 2 in s and s.index(2) < s.index(hi)
        if 9 in s and 15 in s:
            assert s.index(9) < s.index(15)


def test_route_k_equals_E_and_single_expert():
    li = workloads.make_layer("kE", 40, 256, 128, 6, 6, seed=32, wr_std=0.1)
    lg, idx, w = _route(DeviceLayer(li))
    check_routing(li, lg, idx, w)
    assert np.all(np.sort(idx, axis=1) == np.arange(6))
    li1 = workloads.make_layer("E1", 5, 256, 128, 1, 1, seed=33, wr_std=0.1)
    lg, idx, w = _route(DeviceLayer(li1))
    assert np.all(idx == 0) and np.all(w == 1.0)


def test_route_small_token_path():
    # decode sizes take the split-router path when a logits buffer is given
    for T in (1, 4, 16):
        li = workloads.decode(T)
        dl = DeviceLayer(li)
        lg, idx, w = _route(dl)
        check_routing(li, lg, idx, w)


def _prefill_route(li):
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_PREFILL, li.T, li.H, li.I, li.E, li.k)
    dl.prefill(debug=dbg)
    torch.cuda.synchronize()
    return d["logits"].cpu().numpy(), d["topk_idx"].cpu().numpy(), d["topk_w"].cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "prefill", "skewed"])
def test_prefill_routing(name):
    # the prefill forward routes with its own kernels (tensor cores from 128
    # tokens on); its logits, choices and weights meet the same contract
    li = workloads.CONFIGS[name]()
    near = check_routing(li, *_prefill_route(li))
    assert near <= max(2, li.T // 50), f"{near} near-tie tokens"


@pytest.mark.parametrize("T,H,E,k", [
    (128, 256, 2, 1),     # one token tile; three parts of W_r fill less than one box
    (300, 384, 3, 2),     # ragged token tile, E not a multiple of 4
    (260, 256, 256, 8),   # two expert blocks
    (1000, 128, 129, 4),  # one hidden K-block per slice, an expert block of one
])
def test_prefill_routing_shapes(T, H, E, k):
    li = workloads.make_layer("proute", T, H, 128, E, k, seed=T + E, wr_std=0.1)
    check_routing(li, *_prefill_route(li))


@pytest.mark.parametrize("name", ["tiny", "prefill", "skewed"])
def test_bucketing_bit_exact(name):
    li = workloads.CONFIGS[name]()
    dl = DeviceLayer(li)
    d, dbg = moe.make_debug(moe.MOE_MODE_PREFILL, li.T, li.H, li.I, li.E, li.k)
    dl.prefill(debug=dbg)
    torch.cuda.synchronize()
    idx = d["topk_idx"].cpu().numpy()
    off, tok, slot = O.bucket(idx, li.E)
    assert np.array_equal(d["expert_offsets"].cpu().numpy(), off)
    assert np.array_equal(d["bucket_token"].cpu().numpy(), tok)
    assert np.array_equal(d["bucket_slot"].cpu().numpy(), slot)
    # invariants: every token in exactly k buckets, counts sum to T*k
    assert off[-1] == li.T * li.k
    assert np.array_equal(np.bincount(tok, minlength=li.T), np.full(li.T, li.k))
    if name == "skewed":
        # the water-filled Zipf(1.1) popularity of the stored histogram (the
        # oracle's routing; fp32 logits may decide a near tie the other way)
        import test_workloads_skew as SK
        counts = np.diff(off)
        assert np.all(counts[li.notes["dead_experts"]] == 0)
        golden = np.zeros(li.E, np.int64)
        for _, e, n, _ in SK._golden():
            golden[e] = n
        assert np.abs(counts - golden).sum() <= 0.002 * li.T * li.k
