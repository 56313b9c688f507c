"""The whole layer on shapes drawn at random (seeded, so every run checks the
same ones): token counts from 1 to 700, hidden and expert widths of one to
four 128-wide tiles, 8 to 64 experts with top-1 up to top-8, uniform and
skewed logits -- each through the tensor-core kernel (its tile height chosen
by the layer), the CTA-pair kernel and the GEMV kernel (the fused decode
kernel at T <= 8), every output against the oracle with the complete check of
tests/parity.py."""
import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu


def _shapes(n=14, seed=2024):
    r = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        T = int(r.choice([1, 8, int(r.integers(2, 130)), int(r.integers(130, 701)), int(r.integers(130, 701))]))
        H = int(r.choice([128, 256, 384, 512]))
        F = int(r.choice([128, 256, 384]))
        E = int(r.choice([8, 16, 32, 64]))
        k = int(r.integers(1, min(8, E) + 1))
        s = (T, H, E, k, F, bool(r.integers(0, 2)))
        if s not in out:
            out.append(s)
    return out


SHAPES = _shapes()


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


@pytest.mark.parametrize("impl", ["tc", "tc2", "gemv"])
@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: "T{}_H{}_E{}_k{}_F{}{}".format(*s[:5], "_skew" if s[5] else ""))
def test_layer_random_shape(spec, impl):
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    T, H, E, k, F, _ = spec
    d = G.workload(spec, seed=7)
    layer = MoELayerW4(H, E, k, F, d, impl=impl)
    x, logits = G.to_dev_inputs(d)
    out = layer.forward(x, logits).clone()
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    G.check_layer(d, layer, G.bf16_to_f64(out), what=f"random {spec} {impl}")
