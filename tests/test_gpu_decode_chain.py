"""GPU parity of a chain of stacked W4A8 decode layers through the C ABI.

The per-token decode loop of the page "A 35B Hybrid-Attention Mixture-of-
Experts Model on a 6GB 2011 GPU" (Methodology 1, "Decode (CPU)": every
generated token runs through every layer's 4-bit experts): layer l + 1
decodes layer l's bf16 output, each layer a pre-norm residual layer
(MOE_STACKED_PRENORM).  The first 8 layers of the stacked workload (H=2048,
I=768, E=256, top-8, fresh counter-generated Q4_0 weights per layer), one and
four tokens.

Each token is followed along the oracle's own chain (the oracle never sees a
GPU value): while the GPU chose the token's experts as the oracle did, its
layer output must lie within 2e-2 x RMS of the oracle's plus one bf16 ulp
(both sides round to bf16 between layers); where the choice differs, the
oracle's logits must show a near tie, and the token leaves the comparison.
The same chain captured in one CUDA graph and replayed gives the eager
chain's bits.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("bit_quantized_moe_q4_gb300")
from test_gpu_stacked import _gpu_layer  # noqa: E402

L = 8


def _oracle_chain(x_bits):
    S = W.STACK
    xb, hist = x_bits, []
    for l in range(L):
        out, st = O.moe_decode(xb, *W.stacked_layer_lazy(l), S["k"], prenorm=True)
        xb = O.f64_to_bf16_bits(out)
        hist.append((xb, st))
    return hist


@pytest.fixture(scope="module")
def gpu_layers():
    return [_gpu_layer(l, "cuda") for l in range(L)]


@pytest.mark.parametrize("T", [1, 4])
def test_decode_chain_8_layers(gpu_layers, T):
    S = W.STACK
    H, I, E, k = S["H"], S["I"], S["E"], S["k"]
    x0_bits = W.stacked_x()[:T]
    chain = _oracle_chain(x0_bits)
    x0 = torch.from_numpy(x0_bits.view(np.int16)).to("cuda").view(torch.bfloat16)
    ws = torch.empty(moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, T, H, I, E, k),
                     dtype=torch.uint8, device="cuda")
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    idx_bufs = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    dbgs = [moe.MoeDebug(topk_idx=b.data_ptr()) for b in idx_bufs]

    def run(debug):
        x = x0
        for l, (wr, wgu, wd) in enumerate(gpu_layers):
            moe.moe_w4a8_forward_decode(x, wr, wgu, wd, I, k, out=outs[l], out_fp32=False,
                                        workspace=ws, debug=dbgs[l] if debug else None,
                                        prenorm=True)
            x = outs[l]

    run(True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    rows = [o.view(torch.int16).cpu().numpy().view(np.uint16) for o in outs]
    idxs = [b.cpu().numpy().astype(np.int64) for b in idx_bufs]
    compared = 0
    for t in range(T):
        for l in range(L):
            xb_o, st = chain[l]
            if not np.array_equal(idxs[l][t], st["idx"][t]):
                lg = np.sort(st["logits"][t])[::-1]
                gap = float(np.min(lg[:k] - lg[1:k + 1]))
                assert gap < 0.05 * float(np.std(st["logits"][t])), (
                    f"token {t}, layer {l}: experts differ without a near tie (gap {gap:.3g})")
                break
            o = O.bf16_bits_to_f64(xb_o[t])
            g = O.bf16_bits_to_f64(rows[l][t])
            bound = 2e-2 * O.rms(o) + np.abs(o) * 2.0 ** -7
            assert np.all(np.abs(g - o) <= bound), (
                f"token {t}, layer {l}: max|gpu-oracle| {np.max(np.abs(g - o)):.4g}")
            compared += 1
    assert compared >= L * T // 2, f"only {compared} token-layers compared"
    # the whole chain in one graph: the same bits as the eager chain
    eager = [r.copy() for r in rows]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        run(False)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_status() == 0
    for l in range(L):
        assert np.array_equal(outs[l].view(torch.int16).cpu().numpy().view(np.uint16), eager[l])
