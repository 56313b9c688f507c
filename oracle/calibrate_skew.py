"""Fix the bias scale of the skewed long-prefill workload (test infrastructure).

The skewed workload adds beta * (-1.2 * ln rank_e) to every token's logits, the
ranks a seeded permutation of 1..E.  beta is chosen by bisection so that about
30 of the 256 experts receive no assignment at T = 16384 (the configuration's
stated target).  Routing is computed with the oracle only.

Run:  python -m oracle.calibrate_skew   (prints the value stored in workloads.SKEW_BETA)
"""
from __future__ import annotations

import numpy as np

import workloads
from oracle import moe_ref


def empty_experts(beta: float, T: int = 16384, seed: int = 0) -> tuple[int, float]:
    wl = workloads.WORKLOADS["skew16k"]
    tok = workloads.make_tokens(wl.shape, T, seed, skew=True, beta=beta)
    ids, _ = moe_ref.topk_route(tok["logits"], wl.shape.k)
    counts = moe_ref.histogram(ids, wl.shape.E)
    return int((counts == 0).sum()), float(counts.max()) / ids.size


def calibrate(target: int = 30, lo: float = 0.0, hi: float = 4.0, iters: int = 12) -> float:
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        n, _ = empty_experts(mid)
        if n < target:
            lo = mid
        else:
            hi = mid
    return hi


if __name__ == "__main__":
    b = calibrate()
    n, top = empty_experts(b)
    print(f"SKEW_BETA = {b!r}  -> {n} empty experts, hottest expert share {top:.4f}")
