"""The whole layer on the GPU (moe_layer_forward through the C ABI) against the
float64 oracle: every output element within |d| <= 1e-2 + 1e-2*|ref| on
shapes the oracle finishes in seconds, and sampled tokens at full size."""
import numpy as np
import pytest

from oracle import moe_ref

import gpu_util as G

pytestmark = pytest.mark.gpu

IMPLS = ["simt"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_layer(d, impl, block_n=None, reps=1):
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
    (77, 128, 64, 8, 64, False),      # many empty experts
    (1000, 256, 16, 4, 192, True),    # skewed logits (Zipf offset), F not a power of two
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("spec", SMALL, ids=lambda s: "T{}_H{}_E{}_k{}_F{}{}".format(*s[:5], "_skew" if s[5] else ""))
def test_layer_small(spec, impl):
    d = G.workload(spec)
    (got,), _ = run_layer(d, impl)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, spec[3])["out"]
    G.assert_close(got, ref, f"layer {spec} {impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_layer_repeatable(impl):
    """Two calls in a row give the same result (the accumulator is left zero)."""
    d = G.workload((300, 512, 32, 4, 256, False))
    (a, b), _ = run_layer(d, impl, reps=2)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, 4)["out"]
    G.assert_close(a, ref, "first call")
    G.assert_close(b, ref, "second call")


def _sample_tokens(T, n, seed=0):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], r.choice(T, size=min(n, T), replace=False)]))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["decode1", "decode8", "prefill512", "prefill4k", "skew16k"])
def test_layer_full_size_sampled(name, impl):
    """Full-size workloads: every output of a few sampled tokens against the oracle."""
    d = G.workload(name)
    T = d["workload"].T
    (got,), _ = run_layer(d, impl)
    toks = _sample_tokens(T, 6)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, d["workload"].shape.k, tokens=toks)["out"]
    G.assert_close(got[toks], ref, f"{name} sampled tokens {impl}")
    assert np.isfinite(got).all()
