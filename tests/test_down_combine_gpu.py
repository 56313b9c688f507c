"""The down GEMM with the combine in its epilogue (moe_down_combine): the same
bits as the down GEMM followed by moe_combine, its counters left zero after
every call, and the layer built on it passing the oracle check."""
import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

MOE_DEV_BAD_WORKSPACE = 4

CASES = [
    (64, 256, 16, 2, 128, False),     # one tile per expert
    (300, 512, 32, 4, 256, False),    # ragged tiles, several 128-channel blocks per token
    (77, 128, 64, 8, 128, False),     # k = 8, many empty experts, one channel block
    (600, 256, 8, 2, 256, False),     # 128-row tiles: down units of one M-tile
    (1000, 256, 16, 4, 384, True),    # skewed routing
    "prefill512",
    "prefill4k",
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _layers(d):
    from bit_mixture_experts_gb300.layer import MoELayerW4
    s = d["workload"].shape
    fused = MoELayerW4(s.H, s.E, s.k, s.F, d, impl="tc", fuse_combine=True)
    plain = MoELayerW4(s.H, s.E, s.k, s.F, d, impl="tc", fuse_combine=False)
    return fused, plain


@pytest.mark.parametrize("name", CASES, ids=lambda c: c if isinstance(c, str) else "T{}_H{}_E{}_k{}_F{}".format(*c))
def test_fused_combine_equals_two_calls(name):
    """Outputs and y bit for bit those of MOE_DOWN + moe_combine, on two calls in a row (the counters
    return to zero), and the output passes the oracle check (one token per tile at full size)."""
    import torch

    import parity
    from bit_mixture_experts_gb300 import _lib
    d = G.workload(name)
    T = d["workload"].T
    fused, plain = _layers(d)
    x, logits = G.to_dev_inputs(d)
    want = plain.forward(x, logits).clone()
    outs = [fused.forward(x, logits).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    ws = fused.buffers(T)["combine_ws"]
    assert ws is not None and int(ws.count_nonzero().item()) == 0
    for o in outs:
        assert torch.equal(o.view(torch.int16), want.view(torch.int16))
    assert torch.equal(fused.buffers(T)["y"].view(torch.int16), plain.buffers(T)["y"].view(torch.int16))
    got = G.bf16_to_f64(outs[1])
    toks = None
    if isinstance(name, str):
        a = G.gpu_arrays(fused, T, got)
        toks = parity.tile_tokens(a["block_map"], a["num_blocks"], a["perm"], T, d["workload"].shape.k)
    G.check_layer(d, fused, got, tokens=toks, what=f"down+combine {name}")


def test_fused_combine_direct_call_and_bad_workspace():
    """moe_down_combine through the C ABI on the layer's routing and h: the same bits as the two calls;
    a workspace whose counters are not zero is reported (MOE_DEV_BAD_WORKSPACE) and, zeroed again, the
    next call is right."""
    import torch

    from bit_mixture_experts_gb300 import _lib
    spec = (300, 512, 32, 4, 256, False)
    d = G.workload(spec)
    T, H, E, k, F = spec[:5]
    fused, plain = _layers(d)
    x, logits = G.to_dev_inputs(d)
    want = plain.forward(x, logits).clone()
    b = plain.buffers(T)
    bn = plain.block_n_for(T)
    # the layer call may have kept h on chip (moe_expert_ffn_w4): h from the gate/up GEMM on the same routing
    _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_TC, x, T, H, F, E, k, plain.weights.w13, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bn, b["h"])
    ws_bytes = _lib.moe_down_combine_workspace_size(T, H)
    assert ws_bytes == T * (H // 128) * 4
    ws = torch.zeros(ws_bytes // 4, dtype=torch.int32, device=x.device)
    y = torch.empty_like(b["y"])
    out = torch.empty_like(want)
    args = (b["h"], T, H, F, E, k, plain.weights.w2, b["perm"], b["inv_perm"], b["topk_w"], b["block_map"],
            b["num_blocks"], bn, y)
    _lib.moe_down_combine(*args, out, ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert torch.equal(y.view(torch.int16), b["y"].view(torch.int16))
    assert int(ws.count_nonzero().item()) == 0
    # counters above k: every count of the call finds a value above k and reports it (no pair completes)
    ws.fill_(k + 1)
    _lib.moe_down_combine(*args, out, ws)
    assert _lib.moe_get_device_error() == MOE_DEV_BAD_WORKSPACE
    ws.zero_()
    out.zero_()
    _lib.moe_down_combine(*args, out, ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
