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
