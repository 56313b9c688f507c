"""Helpers shared by the GPU parity tests (inputs on the device, library calls)."""
from __future__ import annotations

import functools

import numpy as np

import workloads

TOL_ABS = 1e-2
TOL_REL = 1e-2


def torch_dev():
    import torch
    return torch.device("cuda:0")


def ensure_built():
    from bit_mixture_experts_gb300 import build
    build.build()


@functools.lru_cache(maxsize=4)
def workload(name_or_spec, seed=0):
    """Canonical numpy inputs of a named workload or of a (T, H, E, k, F, skew) tuple."""
    if isinstance(name_or_spec, str):
        return workloads.make_workload(name_or_spec, seed)
    T, H, E, k, F, skew = name_or_spec
    return workloads.make_workload(workloads.custom(T, H, E, k, F, skew), seed)


def to_dev_inputs(d):
    import torch
    dev = torch_dev()
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    return x, logits


def bf16_to_f64(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    tol = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside |d| <= 1e-2 + 1e-2|ref|; "
                             f"worst at {i}: got {got[i]}, ref {ref[i]}")
    return float(err.max())


# statistics of every layer check, printed at the end of the session (tests/conftest.py)
PARITY_STATS = []


def gpu_arrays(layer, T, out, d=None):
    """The GPU's buffers of the last layer call for T tokens, as numpy arrays.  When the call kept h on
    chip (layer.h_on_chip), h is recomputed by the gate/up GEMM alone from the call's routing (needs the
    inputs d), and the down GEMM on that h must give the call's y bit for bit -- so the intermediate
    checks see the h that the fused kernel used."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    b = layer.buffers(T)
    if layer.h_on_chip(T) and d is not None:
        x, _ = to_dev_inputs(d)
        bn = layer.block_n_for(T)
        w = layer.weights
        _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_TC, x, T, layer.H, layer.F, layer.E, layer.k, w.w13,
                                b["perm"], b["topk_w"], b["block_map"], b["num_blocks"], bn, b["h"])
        y2 = torch.empty_like(b["y"])
        _lib.moe_expert_gemm_w4(_lib.DOWN, _lib.IMPL_TC, b["h"], T, layer.H, layer.F, layer.E, layer.k, w.w2,
                                b["perm"], b["topk_w"], b["block_map"], b["num_blocks"], bn, y2)
        torch.cuda.synchronize()
        assert _lib.moe_get_device_error() == 0
        rows = T * layer.k + T
        assert torch.equal(y2[:rows].view(torch.int16), b["y"][:rows].view(torch.int16)), \
            "y of the fused FFN differs from the two GEMMs'"
    return {"topk_ids": b["topk_ids"].cpu().numpy(), "inv_perm": b["inv_perm"].cpu().numpy(),
            "perm": b["perm"].cpu().numpy(), "block_map": b["block_map"].cpu().numpy(),
            "num_blocks": int(b["num_blocks"].item()), "h": bf16_to_f64(b["h"]), "y": bf16_to_f64(b["y"]),
            "out": np.asarray(out, np.float64)}


def check_layer(d, layer, got_out, tokens=None, what=""):
    """Layer parity (tests/parity.py): routing bit-exact, every h and y a valid rounding of its exact
    value, every output within 1e-2 + 1e-2|ref| of the combine on the GPU's y, and of the plain oracle
    except in tokens with a validated rounding flip.  Records and returns the statistics."""
    import parity
    st = parity.check_layer_arrays(d, gpu_arrays(layer, d["workload"].T, got_out, d), tokens=tokens, what=what)
    PARITY_STATS.append((what, st))
    return st
