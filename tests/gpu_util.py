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


H_ABS_BAND = 2e-3     # absolute error allowed on h or y next to zero (cancellation)
H_FLIP_FRAC = 0.01    # at most this share of h (or y) may round away from round-to-nearest


def _check_rounded(gpu_rows, exact_rows, what, name):
    """Every GPU row within one bf16 step of the exact value (or H_ABS_BAND); returns (flips, total)."""
    from oracle import moe_ref
    n_tot = n_flip = 0
    for key, v in exact_rows.items():
        g = gpu_rows(*key)
        lo, hi = moe_ref.bf16_floor_ceil(v)
        band = np.maximum(hi - lo, H_ABS_BAND)
        dev = np.abs(g - v) - band
        assert np.all(dev <= 0), f"{what}: {name} of token {key[0]} expert {key[1]} off by more than one bf16 step"
        n_flip += int((g != moe_ref.round_bf16(v)).sum())
        n_tot += v.size
    assert n_flip <= H_FLIP_FRAC * n_tot, f"{what}: {n_flip} of {n_tot} {name} round away from nearest"
    return n_flip, n_tot


def check_layer(d, layer, got_out, tokens=None, what=""):
    """Layer parity where the bf16 roundings of the intermediates h and y are not unique.

    h = bf16(silu(g) * u) and y = bf16(h Wd^T) round an FP32-accumulated value
    on the GPU and an exact one in the oracle, so a value lying next to a
    rounding midpoint may round to either neighbour.  Checks: (1) every GPU h
    is within one bf16 step of the exact value (or 2e-3 absolute near zero)
    and rounds away from round-to-nearest for at most 1% of elements; (2) the
    same for every GPU y against the exact down projection of the GPU's own h;
    (3) the output equals the oracle's combine evaluated exactly on the GPU's
    own y within |d| <= 1e-2 + 1e-2|ref|, for every element; (4) against the
    plain oracle at least 99% of outputs are within that tolerance.
    Returns a dict of statistics.
    """
    from oracle import moe_ref
    wl = d["workload"]
    s = wl.shape
    T, k, E = wl.T, s.k, s.E
    A = T * k
    b = layer.buffers(T)
    h = bf16_to_f64(b["h"])
    y = bf16_to_f64(b["y"])
    inv = b["inv_perm"].cpu().numpy()
    ids = b["topk_ids"].cpu().numpy()
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, want_h=True)

    def row_of(t, e):
        if e == E:
            return A + t
        j = int(np.nonzero(ids[t] == e)[0][0])
        return inv[t * k + j]

    def gpu_h(t, e):
        return h[row_of(t, e)]

    def gpu_y(t, e):
        return y[row_of(t, e)]

    h_flip, h_tot = _check_rounded(gpu_h, ref["h_exact"], what, "h")
    ref_h = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, h_given=gpu_h, want_y=True)
    y_flip, y_tot = _check_rounded(gpu_y, ref_h["y_exact"], what, "y")
    ref_y = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, y_given=gpu_y)["out"]
    got = np.asarray(got_out)[sel]
    err_y = assert_close(got, ref_y, f"{what} (combine on the GPU's y)")
    err = np.abs(got - ref["out"])
    within = float(np.mean(err <= TOL_ABS + TOL_REL * np.abs(ref["out"])))
    assert within >= 0.99, f"{what}: only {within:.4f} of outputs within tolerance of the plain oracle"
    return {"h_flips": h_flip, "h_total": h_tot, "y_flips": y_flip, "y_total": y_tot, "max_err_given_y": err_y,
            "within_plain": within, "max_err_plain": float(err.max())}
