"""moe_layer_forward_host (host buffers, the end-to-end entry point): the same
bits as moe_layer_forward on device buffers, with pinned host memory (logits
read and out written by the kernels over the host link, x copied) and with
pageable host memory (every buffer copied)."""
import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

CASES = [((64, 256, 16, 2, 128, False), "tc"), ((600, 256, 8, 2, 256, False), "tc"),
         ((5, 256, 16, 4, 128, False), "gemv"), ((1, 256, 16, 2, 128, False), "gemv"),
         ("prefill512", "auto"), ("decode1", "auto")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0] if isinstance(c[0], str) else 'T%d_H%d_E%d_k%d_F%d' % c[0][:5]}-{c[1]}")
def test_forward_host_equals_device(case, pinned):
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    spec, impl = case
    d = G.workload(spec)
    wl = d["workload"]
    s, T = wl.shape, wl.T
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, impl=impl)
    x, logits = G.to_dev_inputs(d)
    want = layer.forward(x, logits).clone()
    xh = torch.from_numpy(d["x_bits"].view(np.int16).copy())
    lh = torch.from_numpy(d["logits"].copy())
    oh = torch.zeros((T, s.H), dtype=torch.int16)
    if pinned:
        xh, lh, oh = xh.pin_memory(), lh.pin_memory(), oh.pin_memory()
    stage = {"x": torch.empty_like(x), "logits": torch.empty_like(logits), "out": torch.zeros_like(want)}
    for _ in range(2):  # twice: the second call starts from the first call's buffers
        layer.forward_host(xh, lh, oh, stage)
        torch.cuda.synchronize()
        assert _lib.moe_get_device_error() == 0
        assert np.array_equal(oh.numpy(), want.view(torch.int16).cpu().numpy())
        oh.zero_()
