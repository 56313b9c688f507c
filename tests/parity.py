"""Layer parity check of the GPU path against the float64 oracle (test infrastructure).

The layer rounds two intermediates to bf16 before the output: h = bf16(silu(g) u)
after the gate/up projection and y = bf16(h Wd^T) after the down projection
(the grouped GEMM writes bf16 rows).  The GPU rounds values accumulated in FP32,
the oracle exact ones, so a value lying next to a rounding midpoint may round to
either neighbour on the GPU: several results are correct there.  The check
therefore compares what is unique and checks that the rest is valid:

1. routing of every checked token is the oracle's (ids bit-exact);
2. every GPU h is the bf16 rounding of some value within delta_h of the exact
   h (computed by the oracle's own dequantised weights), where delta_h bounds
   the FP32 accumulation error (see ``accumulation_bound``); h values that are
   not the round-to-nearest of the exact h are "flips";
3. every GPU y is, in the same sense, a valid rounding of the exact down
   projection of the GPU's own h (delta_y likewise);
4. every output element is within |d| <= 1e-2 + 1e-2 |ref| of the oracle's
   combine evaluated exactly on the GPU's (validated) y rows;
5. every output element is within the same tolerance of the plain oracle
   (``moe_ref.moe_forward`` with no GPU value in it), except in tokens that
   carry at least one validated flip -- those are covered by 2-4, element by
   element.  A miss in a token without a flip fails the check.

The statistics (misses against the plain oracle, flip counts, and how many
misses the h flips alone would cause if y were kept in FP32) are returned so
the tests can report them.

Nothing here is used by the product; it only reads the GPU's outputs as numpy
arrays.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import moe_ref

TOL_ABS = 1e-2
TOL_REL = 1e-2

# Per accumulation step (one K16 MMA, or one add of a warp's partial sum), the
# FP32 rounding error is taken to be at most 2^-20 (eight float32 ulps) of the
# sum of |products| of the dot product, which bounds every partial sum; the
# steps are combined as a random walk (square root of their number).  For the
# GEMM at K = 2048 this allows about 1e-5 of sum |x||w|: ten times what a
# sequential float32 sum of the same products shows on the synthetic inputs.
STEP_ERR = 2.0 ** -20
# Relative error of the FP32 epilogue (silu with the fast exponential and
# division, the product with u, the float32 rounding of g and u).
EPI_REL = 2.0 ** -16


def accumulation_bound(K: int, abs_sum: np.ndarray) -> np.ndarray:
    """Bound on |FP32 result - exact| of dot products of length K with sum |terms| = abs_sum:
    K/16 tensor-core steps plus eight partial sums, STEP_ERR each, as a random walk."""
    steps = K / 16.0 + 8.0
    return STEP_ERR * math.sqrt(steps) * abs_sum


def valid_rounding(gpu: np.ndarray, exact: np.ndarray, delta: np.ndarray):
    """gpu holds bf16 values; valid where gpu = RNE(v) for some v in [exact - delta, exact + delta]
    (RNE is monotone, so that is RNE(exact - delta) <= gpu <= RNE(exact + delta)).
    Returns (valid, flip): flip marks the valid values that differ from RNE(exact)."""
    lo = moe_ref.round_bf16(exact - delta)
    hi = moe_ref.round_bf16(exact + delta)
    valid = (gpu >= lo) & (gpu <= hi) & np.isfinite(gpu)
    flip = valid & (gpu != moe_ref.round_bf16(exact))
    return valid, flip


def silu_and_slope(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return g * s, s * (1.0 + g * (1.0 - s))


def check_layer_arrays(d: dict, gpu: dict, tokens=None, what: str = "") -> dict:
    """Check the GPU's layer call on the workload ``d`` (numpy arrays of the GPU's buffers:
    topk_ids [T,k], inv_perm [A], h [A+T,F], y [A+T,H], out [T,H], values as float64)
    for the tokens ``tokens`` (all by default).  Raises AssertionError on a failure;
    returns statistics."""
    wl = d["workload"]
    s = wl.shape
    T, H, E, k, F = wl.T, s.H, s.E, s.k, s.F
    A = T * k
    sel = np.arange(T) if tokens is None else np.unique(np.asarray(tokens, dtype=np.int64))
    n = sel.size
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, tokens=sel, want_h=True)
    ids, w = ref["topk_ids"], ref["topk_w"]
    gids = np.asarray(gpu["topk_ids"])[sel]
    assert np.array_equal(gids, ids), f"{what}: routing ids differ from the oracle's"
    inv = np.asarray(gpu["inv_perm"])
    gh, gy = gpu["h"], gpu["y"]
    got = np.asarray(gpu["out"], dtype=np.float64)[sel]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    x = moe_ref.bf16_value(np.asarray(d["x_bits"])[sel])

    acc_gy = np.zeros((n, H))      # combine on the GPU's y
    acc_f32y_gpu = np.zeros((n, H))  # the GPU's h, y kept unrounded (statistics only)
    acc_f32y_ref = np.zeros((n, H))  # the oracle's h, y kept unrounded (statistics only)
    flip_tok = np.zeros(n, dtype=bool)
    st = {"h_total": 0, "h_flips": 0, "y_total": 0, "y_flips": 0, "h_delta_ulp_max": 0.0}
    for e in sorted(set(np.unique(ids).tolist()) | {E}):
        if e == E:
            idx, wt = np.arange(n), np.ones(n)
            rows = A + sel
        else:
            idx, cols = np.nonzero(ids == e)
            wt = w[idx, cols]
            rows = inv[sel[idx] * k + cols]
        assert np.all((rows >= 0) & (rows < A + T)), f"{what}: inv_perm out of range"
        w13, w2 = moe_ref.expert_weights(d, e)
        xr = x[idx]
        g = xr @ w13[:F].T
        u = xr @ w13[F:].T
        h_exact = np.stack([ref["h_exact"][(int(sel[i]), int(e))] for i in idx])
        silu_g, slope = silu_and_slope(g)
        eg = accumulation_bound(H, np.abs(xr) @ np.abs(w13[:F]).T)
        eu = accumulation_bound(H, np.abs(xr) @ np.abs(w13[F:]).T)
        d_h = np.abs(slope * u) * eg + np.abs(silu_g) * eu + EPI_REL * np.abs(h_exact)
        hg = np.asarray(gh[rows], dtype=np.float64)
        ok, fl = valid_rounding(hg, h_exact, d_h)
        if not ok.all():
            i, f = np.argwhere(~ok)[0]
            raise AssertionError(f"{what}: h of token {sel[idx[i]]} expert {e} feature {f}: GPU {hg[i, f]!r}, "
                                 f"exact {h_exact[i, f]!r}, allowed accumulation error {d_h[i, f]:.3g} "
                                 f"({int((~ok).sum())} invalid h values for this expert)")
        lo, hi = moe_ref.bf16_floor_ceil(h_exact)
        ulp = np.where(hi > lo, hi - lo, 1.0)
        st["h_delta_ulp_max"] = max(st["h_delta_ulp_max"], float((d_h / ulp).max()))
        y_exact = hg @ w2.T
        d_y = accumulation_bound(F, np.abs(hg) @ np.abs(w2).T)
        yg = np.asarray(gy[rows], dtype=np.float64)
        oky, fly = valid_rounding(yg, y_exact, d_y)
        if not oky.all():
            i, c = np.argwhere(~oky)[0]
            raise AssertionError(f"{what}: y of token {sel[idx[i]]} expert {e} channel {c}: GPU {yg[i, c]!r}, "
                                 f"exact down projection of the GPU's h {y_exact[i, c]!r}, allowed "
                                 f"accumulation error {d_y[i, c]:.3g} ({int((~oky).sum())} invalid y values)")
        acc_gy[idx] += wt[:, None] * yg
        acc_f32y_gpu[idx] += wt[:, None] * y_exact
        acc_f32y_ref[idx] += wt[:, None] * (moe_ref.round_bf16(h_exact) @ w2.T)
        flip_tok[idx] |= fl.any(1) | fly.any(1)
        st["h_total"] += hg.size
        st["h_flips"] += int(fl.sum())
        st["y_total"] += yg.size
        st["y_flips"] += int(fly.sum())

    tol = lambda ref_: TOL_ABS + TOL_REL * np.abs(ref_)  # noqa: E731
    out_gy = moe_ref.round_bf16(acc_gy)
    bad_gy = np.abs(got - out_gy) > tol(out_gy)
    if bad_gy.any():
        i, c = np.argwhere(bad_gy)[0]
        raise AssertionError(f"{what}: {int(bad_gy.sum())} outputs differ from the combine of the GPU's y rows; "
                             f"first token {sel[i]} channel {c}: got {got[i, c]!r}, ref {out_gy[i, c]!r}")
    plain = ref["out"]
    miss = np.abs(got - plain) > tol(plain)
    miss_tok = miss.any(1)
    unexplained = miss_tok & ~flip_tok
    if unexplained.any():
        i = int(np.nonzero(unexplained)[0][0])
        c = int(np.nonzero(miss[i])[0][0])
        raise AssertionError(f"{what}: token {sel[i]} has {int(miss[i].sum())} outputs outside 1e-2 + 1e-2|ref| of "
                             f"the plain oracle and no h or y rounding flip to explain them; channel {c}: got "
                             f"{got[i, c]!r}, oracle {plain[i, c]!r}")
    f32_gpu = moe_ref.round_bf16(acc_f32y_gpu)
    f32_ref = moe_ref.round_bf16(acc_f32y_ref)
    st.update({
        "tokens": int(n), "outputs": int(got.size), "misses_plain": int(miss.sum()),
        "within_plain": float(1.0 - miss.mean()), "miss_tokens": int(miss_tok.sum()),
        "flip_tokens": int(flip_tok.sum()),
        "misses_if_y_fp32": int((np.abs(f32_gpu - f32_ref) > tol(f32_ref)).sum()),
        "max_err_plain": float(np.abs(got - plain).max()),
        "max_err_given_y": float(np.abs(got - out_gy).max()),
    })
    return st


def summary_line(name: str, st: dict) -> str:
    return (f"{name}: {st['outputs']} outputs of {st['tokens']} tokens; plain oracle: {st['misses_plain']} outside "
            f"tol in {st['miss_tokens']} tokens (all with validated flips; {st['flip_tokens']} tokens have one); "
            f"h flips {st['h_flips']}/{st['h_total']}, y flips {st['y_flips']}/{st['y_total']}; "
            f"misses if y were FP32 {st['misses_if_y_fp32']}; max |d| plain {st['max_err_plain']:.3g}")


def tile_tokens(block_map: np.ndarray, num_blocks: int, perm: np.ndarray, T: int, k: int) -> np.ndarray:
    """One token per block-map tile: the token of the tile's last row (plus tokens 0 and T-1), so a
    check of these tokens' outputs touches every tile, ragged tails included."""
    A = T * k
    bm = np.asarray(block_map)[:num_blocks]
    last = bm[:, 1] + bm[:, 2] - 1
    toks = np.where(last >= A, last - A, np.asarray(perm)[np.minimum(last, A - 1)] // k)
    return np.unique(np.concatenate([toks, [0, T - 1]]))
