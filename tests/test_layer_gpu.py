"""The whole layer on the GPU (moe_layer_forward through the C ABI) against the
float64 oracle: every output element within |d| <= 1e-2 + 1e-2*|ref| on
shapes the oracle finishes in seconds, and sampled tokens at full size."""
import numpy as np
import pytest

from oracle import moe_ref

import gpu_util as G

pytestmark = pytest.mark.gpu

IMPLS = ["tc", "simt", "gemv"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_layer(d, impl, block_n=None, reps=1):
    """Layer forward(s) through the C ABI; returns the outputs (float64) and the layer."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    wl = d["workload"]
    s = wl.shape
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, impl=impl, block_n=block_n)
    x, logits = G.to_dev_inputs(d)
    outs = []
    for _ in range(reps):
        outs.append(layer.forward(x, logits).clone())
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    return [G.bf16_to_f64(o) for o in outs], layer


SMALL = [
    (64, 256, 16, 2, 128, False),     # the tiny workload's shape
    (300, 512, 32, 4, 256, False),    # ragged tiles, several shared-expert tiles
    (512, 256, 8, 2, 128, False),     # experts above one tile
    (1, 256, 16, 2, 128, False),      # a single token
    (77, 128, 64, 8, 128, False),     # many empty experts
    (1000, 256, 16, 4, 384, True),    # skewed logits (Zipf offset), F not a power of two
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("spec", SMALL, ids=lambda s: "T{}_H{}_E{}_k{}_F{}{}".format(*s[:5], "_skew" if s[5] else ""))
def test_layer_small(spec, impl):
    d = G.workload(spec)
    (got,), layer = run_layer(d, impl)
    G.check_layer(d, layer, got, what=f"layer {spec} {impl}")


@pytest.mark.parametrize("block_n", [16, 48, 64, 96, 128])
def test_layer_tc_block_sizes(block_n):
    """The tensor-core kernel with every tile height it supports (N = rows rounded up to 16)."""
    spec = (700, 256, 16, 4, 128, False)
    d = G.workload(spec)
    (got,), layer = run_layer(d, "tc", block_n=block_n)
    G.check_layer(d, layer, got, what=f"tc block_n={block_n}")


def test_layer_simt_odd_widths():
    """The CUDA-core kernel covers widths the tensor-core one does not take (F % 128 != 0)."""
    for spec in [(77, 128, 64, 8, 64, False), (300, 256, 16, 4, 192, True)]:
        d = G.workload(spec)
        (got,), layer = run_layer(d, "simt")
        G.check_layer(d, layer, got, what=f"simt {spec}")


@pytest.mark.parametrize("impl", IMPLS)
def test_layer_repeatable(impl):
    """Two calls in a row give the same result (the accumulator is left zero)."""
    d = G.workload((300, 512, 32, 4, 256, False))
    (a, b), layer = run_layer(d, impl, reps=2)
    G.check_layer(d, layer, a, what="first call")
    G.check_layer(d, layer, b, what="second call")


def _sample_tokens(T, n, seed=0):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], r.choice(T, size=min(n, T), replace=False)]))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["decode1", "decode8", "prefill512", "prefill4k", "skew16k"])
def test_layer_full_size_sampled(name, impl):
    """Full-size workloads: every output of a few sampled tokens against the oracle."""
    d = G.workload(name)
    T = d["workload"].T
    (got,), layer = run_layer(d, impl)
    toks = _sample_tokens(T, 6)
    G.check_layer(d, layer, got, tokens=toks, what=f"{name} sampled tokens {impl}")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("impl", IMPLS)
def test_gate_up_intermediate(impl):
    """The gate/up GEMM alone: h = bf16(silu(g) u) per permuted row against the oracle's h."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    spec = (200, 256, 8, 2, 128, False)
    d = G.workload(spec)
    T, H, E, k, F = spec[:5]
    layer = MoELayerW4(H, E, k, F, d, impl=impl)
    x, logits = G.to_dev_inputs(d)
    b = layer.buffers(T)
    w = layer.weights
    bn = layer.block_n_for(T)
    _lib.moe_route(logits, k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                   b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
    b["h"].zero_()
    _lib.moe_expert_gemm_w4(_lib.GATE_UP, layer.impl_for(T), x, T, H, F, E, k, w.w13, w.s13, w.b13, b["perm"],
                            b["topk_w"], b["block_map"], b["num_blocks"], bn, b["h"])
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    got = G.bf16_to_f64(b["h"])
    perm = b["perm"].cpu().numpy()
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, want_h=True)
    ids = ref["topk_ids"].ravel()
    A = T * k
    want = np.zeros((A + T, F))
    for r in range(A):
        a = int(perm[r])
        want[r] = ref["h"][(a // k, int(ids[a]))]
    exact = np.zeros((A + T, F))
    for r in range(A):
        a = int(perm[r])
        exact[r] = ref["h_exact"][(a // k, int(ids[a]))]
    for t in range(T):
        want[A + t] = ref["h"][(t, E)]
        exact[A + t] = ref["h_exact"][(t, E)]
    lo, hi = moe_ref.bf16_floor_ceil(exact)
    assert np.all(np.abs(got - exact) <= np.maximum(hi - lo, G.H_ABS_BAND)), f"h {impl}"
    assert (got != want).mean() <= G.H_FLIP_FRAC, f"h {impl}: too many roundings away from nearest"
