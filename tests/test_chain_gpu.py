"""The decode chain (layer.MoEDecodeChain): several MoE layers in sequence, each
layer's input the RMS norm of the previous layer's output and its logits the
router projection of that input, on the GPU.  Every layer is checked against
the oracle on the GPU's own data of the step before (the previous layer's
output, itself checked): the norm a valid bf16 rounding of the exact one, the
logits within the FP32 accumulation bound of the exact projection, the routing
equal to the oracle's routing of those logits bit for bit, and the output with
the complete layer check of tests/parity.py."""
import math

import numpy as np
import pytest

import workloads
from oracle import moe_ref

import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _chain_check(T, shape, L, what):
    import parity
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoEDecodeChain
    H, E, k, F = shape.H, shape.E, shape.k, shape.F
    ws = [workloads.make_weights(shape, seed=10 + l) for l in range(L)]
    wrs = [workloads.router_weight_bits(shape, seed=10 + l) for l in range(L)]
    chain = MoEDecodeChain(H, E, k, F, ws, wrs, device=G.torch_dev(), impl="gemv")
    tok = workloads.make_tokens(shape, T, seed=9)
    x0 = torch.from_numpy(tok["x_bits"].view(np.int16)).to(G.torch_dev()).view(torch.bfloat16)
    chain.forward(x0)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    b = chain.buffers(T)
    prev = tok["x_bits"]
    wl = workloads.custom(T, H, E, k, F)
    for l in range(L):
        # the norm of the previous output: a valid rounding of the exact value, allowing the FP32 sum of
        # squares (H/32 terms per lane, then five shuffle levels) and the scale's three roundings
        x_bits = b["xn"][l].view(torch.int16).cpu().numpy().view(np.uint16)
        pv = moe_ref.bf16_value(prev)
        exact_n = pv / np.sqrt(np.mean(pv * pv, axis=-1, keepdims=True) + moe_ref.RMS_EPS)
        rel = (H / 32 + 16) * 2.0 ** -24
        ok, _ = parity.valid_rounding(moe_ref.bf16_value(x_bits), exact_n, rel * np.abs(exact_n))
        assert ok.all(), f"{what} layer {l}: {int((~ok).sum())} normalised inputs are not a rounding of the exact"
        logits = b["logits"][l].cpu().numpy()
        exact = moe_ref.router_logits(x_bits, wrs[l]).astype(np.float64)
        xv, wv = moe_ref.bf16_value(x_bits), moe_ref.bf16_value(wrs[l])
        bound = 2.0 ** -20 * math.sqrt(H / 16 + 8) * (np.abs(xv) @ np.abs(wv).T) + np.abs(exact) * 2.0 ** -24
        assert np.all(np.abs(logits - exact) <= bound), f"{what} layer {l}: logits beyond the bound"
        layer = chain.layers[l]
        lb = layer.buffers(T)
        ref = moe_ref.route(logits, k, layer.block_n_for(T))
        assert np.array_equal(lb["topk_ids"].cpu().numpy(), ref["topk_ids"]), f"{what} layer {l}: routing"
        d = dict(ws[l])
        d.update({"workload": wl, "x_bits": x_bits, "logits": logits})
        out = G.bf16_to_f64(b["out"][l])
        st = parity.check_layer_arrays(d, G.gpu_arrays(layer, T, out), what=f"{what} layer {l}")
        G.PARITY_STATS.append((f"{what} layer {l}", st))
        prev = b["out"][l].view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T", [1, 5, 8])
def test_chain_small(T):
    _chain_check(T, workloads.LayerShape(H=256, E=64, k=4, F=128), 3, f"chain T={T}")


def test_chain_full_width_batch1():
    _chain_check(1, workloads.FULL, 2, "chain full width T=1")


@pytest.mark.parametrize("T,H,E", [(1, 2048, 256), (8, 256, 64), (5, 128, 8), (3, 136, 17)])
def test_norm_router_equals_rms_norm(T, H, E):
    """moe_norm_router's normalised input is bit for bit moe_rms_norm's, and its logits are within the
    FP32 accumulation bound of the exact projection of that input (H = 136 and E = 17: sizes that
    are no multiple of a warp's 32 lanes of 8-element chunks, or of the kernel's experts per CTA)."""
    import torch

    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    shape = workloads.LayerShape(H=H, E=E, k=min(4, E), F=128)
    tok = workloads.make_tokens(shape, T, seed=21)
    wr = workloads.router_weight_bits(shape, seed=22)
    x = torch.from_numpy(tok["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    w = torch.from_numpy(wr.view(np.int16)).to(dev).view(torch.bfloat16)
    xn1 = torch.empty_like(x)
    xn2 = torch.empty_like(x)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    _lib.moe_rms_norm(x, xn1)
    _lib.moe_norm_router(x, w, xn2, logits)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    assert torch.equal(xn1.view(torch.int16), xn2.view(torch.int16))
    x_bits = xn2.view(torch.int16).cpu().numpy().view(np.uint16)
    exact = moe_ref.router_logits(x_bits, wr).astype(np.float64)
    xv, wv = moe_ref.bf16_value(x_bits), moe_ref.bf16_value(wr)
    bound = 2.0 ** -20 * math.sqrt(H / 16 + 8) * (np.abs(xv) @ np.abs(wv).T) + np.abs(exact) * 2.0 ** -24
    assert np.all(np.abs(logits.cpu().numpy() - exact) <= bound)
