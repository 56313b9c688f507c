"""Failure detection without a GPU fault: a wait limit far below the time the
kernels' waits take makes them run out.  The layer call must come back with
MOE_DEV_TIMEOUT in the device error word (no hang, no trap), and the same
context must give correct results again once the limit is restored.

Collected after the other layer tests (file name) and the short limit is
restored in a finally block, so it cannot leak into other tests."""
import numpy as np
import pytest

import gpu_util as G

pytestmark = pytest.mark.gpu

MOE_DEV_TIMEOUT = 3
DEFAULT_LIMIT_NS = 1_000_000_000


@pytest.mark.parametrize("impl", ["tc", "gemv", "ffn"])
def test_wait_timeout_reported_and_recovered(impl):
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    G.ensure_built()
    # tc: 300 tokens (multi-CTA routing with its grid barrier, pipeline waits of the GEMM);
    # gemv: 8 tokens (the fused decode kernel and its grid barriers)
    # ffn: 200 tokens with F = 256 (64-row tiles: both projections in one launch, h kept on chip)
    spec = {"tc": (300, 256, 16, 4, 128, False), "gemv": (8, 256, 16, 4, 128, False),
            "ffn": (200, 256, 16, 4, 256, False)}[impl]
    d = G.workload(spec)
    T, H, E, k, F, _ = spec
    layer = MoELayerW4(H, E, k, F, d, impl="tc" if impl == "ffn" else impl)
    assert layer.h_on_chip(T) == (impl == "ffn")
    x, logits = G.to_dev_inputs(d)
    good = layer.forward(x, logits).clone()
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    # 0.2 us: a wait on memory or another CTA that is still open after its first check runs out
    # (limits this short are polled, not slept on, so they are checked on time).  Whether a wait
    # stays open that long depends on timing (the CTAs of a grid barrier can arrive within the
    # limit), so the call is repeated (the device error word is read and cleared after each) until
    # a timeout is reported.
    _lib.moe_set_wait_limit_ns(200)
    code = 0
    try:
        for _ in range(20):
            layer.forward(x, logits)
            torch.cuda.synchronize()
            code = _lib.moe_get_device_error()
            if code:
                break
    finally:
        _lib.moe_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    assert code == MOE_DEV_TIMEOUT, code
    # the context still works and the results are right again
    again = layer.forward(x, logits)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    assert np.array_equal(G.bf16_to_f64(again), G.bf16_to_f64(good))
