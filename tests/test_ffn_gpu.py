"""Both projections of every expert tile in one launch with h kept on chip
(moe_expert_ffn_w4, which the layer call uses for tiles of at most 64 rows):
y and the layer output bit for bit those of the two grouped GEMMs with h
through HBM, on shapes with several tiles per expert, ragged tails, k = 8,
skewed routing and the full-width 512-token prefill; the output also passes
the oracle check."""
import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

CASES = [
    ((64, 256, 16, 2, 256, False), None),
    ((300, 512, 32, 4, 256, False), None),
    ((600, 256, 8, 2, 256, False), 64),      # 64-row tiles, several per expert
    ((77, 128, 64, 8, 256, False), 32),      # k = 8, many empty experts, 32-row tiles
    ((1000, 256, 16, 4, 512, True), 48),     # skewed routing, 48-row tiles (ragged N)
    ((9, 256, 8, 2, 256, False), 16),        # 16-row tiles
    ("prefill512", None),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


@pytest.mark.parametrize("case", CASES, ids=lambda c: (c[0] if isinstance(c[0], str) else "T{}_H{}_E{}_k{}_F{}".format(*c[0][:5])) + f"_bn{c[1]}")
def test_fused_ffn_equals_two_gemms(case):
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    spec, bn = case
    d = G.workload(spec)
    wl = d["workload"]
    s, T = wl.shape, wl.T
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, impl="tc", block_n=bn)
    assert layer.h_on_chip(T)
    x, logits = G.to_dev_inputs(d)
    outs = [layer.forward(x, logits).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    b = layer.buffers(T)
    y_fused = b["y"].clone()
    # the two grouped GEMMs on the same routing, h through HBM, then the same combine
    bnt = layer.block_n_for(T)
    w = layer.weights
    h = torch.empty_like(b["h"])
    y = torch.empty_like(b["y"])
    out = torch.empty_like(outs[0])
    _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_TC, x, T, s.H, s.F, s.E, s.k, w.w13, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bnt, h)
    _lib.moe_expert_gemm_w4(_lib.DOWN, _lib.IMPL_TC, h, T, s.H, s.F, s.E, s.k, w.w2, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bnt, y)
    _lib.moe_combine(y, b["inv_perm"], b["topk_w"], out)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    rows = T * s.k + T
    assert torch.equal(y_fused[:rows].view(torch.int16), y[:rows].view(torch.int16))
    for o in outs:
        assert torch.equal(o.view(torch.int16), out.view(torch.int16))
    G.check_layer(d, layer, G.bf16_to_f64(outs[1]), what=f"fused FFN {spec}")
