"""moe_route_x on the GPU: the router projection (bf16 x times bf16 router rows,
FP32 accumulation on the tensor cores) fused with the top-k, then routing,
against the oracle.  Small-integer operands make every logit exact, so logits
and routing must equal the oracle's bit for bit.  On random operands every
logit must be within the FP32 accumulation bound of the exact one; the routing
must equal the oracle's routing of the GPU's own logits bit for bit (the
decision taken in the same precision), and the chosen experts must be a valid
top-k of the exact logits (any difference is a near-tie within the bound)."""
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


def _run(x_bits, wr_bits, k, bn):
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    T, H = x_bits.shape
    E = wr_bits.shape[0]
    A = T * k
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev)
    w = torch.from_numpy(np.ascontiguousarray(wr_bits).view(np.int16)).to(dev)
    cap = _lib.moe_block_map_capacity(T, E, k, bn)
    b = {"logits": torch.full((T, E), float("nan"), dtype=torch.float32, device=dev),
         "topk_ids": torch.full((T, k), -7, dtype=torch.int32, device=dev),
         "topk_w": torch.zeros((T, k), dtype=torch.float32, device=dev),
         "counts": torch.empty(E, dtype=torch.int32, device=dev),
         "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "perm": torch.empty(A, dtype=torch.int32, device=dev),
         "inv_perm": torch.empty(A, dtype=torch.int32, device=dev),
         "block_map": torch.empty((cap, 3), dtype=torch.int32, device=dev),
         "num_blocks": torch.empty(1, dtype=torch.int32, device=dev)}
    ws = torch.zeros(max(_lib.moe_route_workspace_size(T, E, k, bn), 16), dtype=torch.uint8, device=dev)
    _lib.moe_route_x(x, w, k, bn, *(b[n] for n in ("logits", "topk_ids", "topk_w", "counts", "offsets", "perm",
                                                   "inv_perm", "block_map", "num_blocks")), ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    return {n: v.cpu().numpy() for n, v in b.items()}


def _check_routing(got, logits, k, bn):
    ref = moe_ref.route(logits, k, bn)
    for n in ("topk_ids", "counts", "offsets", "perm", "inv_perm"):
        assert np.array_equal(got[n], ref[n]), n
    nb = int(got["num_blocks"][0])
    assert nb == ref["num_blocks"]
    assert np.array_equal(got["block_map"][:nb], ref["block_map"])
    assert np.allclose(got["topk_w"], ref["topk_w"], rtol=1e-6, atol=float(np.finfo(np.float32).tiny))


@pytest.mark.parametrize("T,H,E,k", [(5, 192, 64, 4), (130, 256, 128, 8), (300, 512, 256, 8)])
def test_route_x_exact_on_integer_operands(T, H, E, k):
    r = np.random.default_rng(T + H + E)
    xb = workloads.f32_to_bf16_bits(r.integers(-3, 4, size=(T, H)).astype(np.float32))
    wb = workloads.f32_to_bf16_bits(r.integers(-2, 3, size=(E, H)).astype(np.float32))
    got = _run(xb, wb, k, 128)
    ref = moe_ref.router_logits(xb, wb)
    assert np.array_equal(got["logits"], ref)
    _check_routing(got, ref, k, 128)


@pytest.mark.parametrize("T,H,E,k,bn", [(1, 2048, 256, 8, 8), (64, 256, 64, 2, 128), (512, 2048, 256, 8, 64),
                                        (777, 1024, 512, 16, 128), (4096, 2048, 256, 8, 128)])
def test_route_x_random(T, H, E, k, bn):
    shape = workloads.LayerShape(H=H, E=E, k=k, F=128)
    tok = workloads.make_tokens(shape, T, seed=3)
    xb = tok["x_bits"]
    wb = workloads.router_weight_bits(shape, seed=3)
    got = _run(xb, wb, k, bn)
    exact = moe_ref.router_logits(xb, wb).astype(np.float64)
    x = moe_ref.bf16_value(xb)
    w = moe_ref.bf16_value(wb)
    bound = 2.0 ** -20 * math.sqrt(H / 16 + 8) * (np.abs(x) @ np.abs(w).T) + np.abs(exact) * 2.0 ** -24
    err = np.abs(got["logits"].astype(np.float64) - exact)
    assert np.all(err <= bound), f"{int((err > bound).sum())} logits beyond the FP32 accumulation bound"
    # the decision on the GPU's own float32 logits is the oracle's, bit for bit
    _check_routing(got, got["logits"], k, bn)
    # and it is a valid top-k of the exact logits: whatever it leaves out is no larger than what it
    # keeps, except within the bound (near-ties)
    ids = got["topk_ids"].astype(np.int64)
    for t in range(T):
        chosen = exact[t, ids[t]]
        rest = np.delete(exact[t], ids[t])
        if rest.size:
            assert rest.max() <= chosen.min() + 2 * bound[t].max(), t
    print(f"route_x T={T} H={H} E={E} k={k}: max |logit - exact| {err.max():.3g}, "
          f"{int((err > 0).sum())} of {err.size} logits not equal to the exactly rounded sum")
