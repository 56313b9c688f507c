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


H_ABS_BAND = 2e-3     # absolute error allowed on h next to zero (cancellation in g or u)
H_FLIP_FRAC = 0.01    # at most this share of h may round away from round-to-nearest


def check_layer(d, layer, got_out, tokens=None, what=""):
    """Layer parity where the bf16 rounding of the intermediate h is not unique.

    h = bf16(silu(g) * u) rounds an FP32-accumulated value on the GPU and an
    exact one in the oracle, so an h lying next to a rounding midpoint may
    round to either neighbour.  Checks: (1) every GPU h is within one bf16 step
    of the exact value (or 2e-3 absolute near zero) and rounds away from
    round-to-nearest for at most 1% of elements; (2) the output equals the
    oracle's down projection + combine evaluated exactly on the GPU's own h
    within |d| <= 1e-2 + 1e-2|ref|, for every element; (3) against the plain
    oracle at least 99% of outputs are within that tolerance.
    Returns a dict of statistics.
    """
    from oracle import moe_ref
    wl = d["workload"]
    s = wl.shape
    T, k, E = wl.T, s.k, s.E
    A = T * k
    b = layer.buffers(T)
    h = bf16_to_f64(b["h"])
    inv = b["inv_perm"].cpu().numpy()
    ids = b["topk_ids"].cpu().numpy()
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, want_h=True)

    def gpu_h(t, e):
        if e == E:
            return h[A + t]
        j = int(np.nonzero(ids[t] == e)[0][0])
        return h[inv[t * k + j]]

    n_h = n_flip = 0
    worst = 0.0
    for (t, e), v in ref["h_exact"].items():
        g = gpu_h(t, e)
        lo, hi = moe_ref.bf16_floor_ceil(v)
        band = np.maximum(hi - lo, H_ABS_BAND)
        dev = np.abs(g - v) - band
        worst = max(worst, float(dev.max()))
        assert np.all(dev <= 0), f"{what}: h of token {t} expert {e} off by more than one bf16 step"
        n_flip += int((g != moe_ref.round_bf16(v)).sum())
        n_h += v.size
    assert n_flip <= H_FLIP_FRAC * n_h, f"{what}: {n_flip} of {n_h} h round away from nearest"
    ref_g = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, h_given=gpu_h)["out"]
    got = np.asarray(got_out)[sel]
    err_g = assert_close(got, ref_g, f"{what} (down+combine on the GPU's h)")
    err = np.abs(got - ref["out"])
    within = float(np.mean(err <= TOL_ABS + TOL_REL * np.abs(ref["out"])))
    assert within >= 0.99, f"{what}: only {within:.4f} of outputs within tolerance of the plain oracle"
    return {"h_flips": n_flip, "h_total": n_h, "max_err_given_h": err_g, "within_plain": within,
            "max_err_plain": float(err.max())}
