"""Wait statistics of the tensor-core kernels on one workload (trace build).

    python -m bit_mixture_experts_gb300.trace [--workload prefill4k] [--block-n N] [--json]

Builds libmoe_w4_trace.so (-DMOE_TRACE) if it is missing or stale and loads it
in place of libmoe_w4.so, runs the layer once on the workload's synthetic
inputs (routing, buffers), then launches each grouped kernel of the layer's
path once more by itself between moe_trace_reset and moe_trace_read: the fused
expert FFN (moe_expert_ffn_w4) where the layer keeps h on chip, else the gate/up
and the down GEMM (moe_expert_gemm_w4).  For every role of the kernel's warps
it prints the share of the role's span spent in the kernel's bounded mbarrier
waits (median over the CTAs), the waits per warp, and the spread of the CTAs'
spans.  What a role does between its waits -- issuing MMAs, expanding
weights, converting accumulators -- is the rest of its span.

Run from the repository root (the workload generators live in `workloads`).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

from . import _lib, build

# warp roles of gemm_tc_kernel and ffn_tc_kernel (512 threads, one CTA per SM)
ROLES = [("weight producer", range(0, 1)), ("MMA issuer", range(1, 2)), ("activation loads", range(2, 4)),
         ("dequantisation", range(4, 12)), ("epilogue", range(12, 16))]
TRACE_CTAS = 1024


def role_stats(words: np.ndarray, ctas: int) -> dict:
    """Per-role statistics from the trace words of one launch ([1024, 32, 4] uint64: cycles waited,
    waits, the complement of the first wait's start, the last wait's end, per CTA and warp)."""
    u = words.reshape(TRACE_CTAS, 32, 4)[:ctas].copy()
    u[:, :, 2] = np.where(u[:, :, 1] > 0, ~u[:, :, 2], 0)  # back to clock64, in integers
    t = u.astype(np.float64)
    out = {}
    for name, warps in ROLES:
        w = t[:, list(warps), :]
        live = w[:, :, 1].sum(axis=1) > 0
        if not live.any():
            continue
        w = w[live]
        first = np.where(w[:, :, 1] > 0, w[:, :, 2], np.inf).min(axis=1)
        last = w[:, :, 3].max(axis=1)
        span = np.maximum(last - first, 1.0)
        share = w[:, :, 0].sum(axis=1) / (len(warps) * span)
        out[name] = {"warps": len(warps), "ctas": int(live.sum()),
                     "wait_share_median": float(np.median(share)), "wait_share_min": float(share.min()),
                     "wait_share_max": float(share.max()),
                     "waits_per_warp": float(np.median(w[:, :, 1].sum(axis=1) / len(warps))),
                     "span_kcycles_min": float(span.min() / 1e3), "span_kcycles_median": float(np.median(span) / 1e3),
                     "span_kcycles_max": float(span.max() / 1e3)}
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="prefill4k")
    ap.add_argument("--block-n", type=int, default=None)
    ap.add_argument("--json", action="store_true", help="print one JSON object instead of the table")
    a = ap.parse_args(argv)

    sys.path.insert(0, os.getcwd())
    import torch
    import workloads
    lib_path = build.build(trace=True)
    _lib.load(lib_path)  # every wrapper of _lib now calls the trace build
    if _lib.moe_trace_words() == 0:
        raise RuntimeError(f"{lib_path} records no wait statistics")
    from .layer import MoELayerW4

    d = workloads.make_workload(a.workload, 0)
    s, T = d["workload"].shape, d["workload"].T
    dev = torch.device("cuda:0")
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, device=dev, impl="tc", block_n=a.block_n)
    bn = layer.block_n_for(T)
    layer.forward(x, logits)
    torch.cuda.synchronize()
    b, w = layer.buffers(T), layer.weights
    if layer.h_on_chip(T):
        calls = [("ffn_tc_kernel (fused expert FFN)",
                  lambda: _lib.moe_expert_ffn_w4(x, T, s.H, s.F, s.E, s.k, w.w13, w.w2, b["perm"], b["block_map"],
                                                 b["num_blocks"], bn, b["y"]))]
    else:
        calls = [("gemm_tc_kernel gate/up",
                  lambda: _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_TC, x, T, s.H, s.F, s.E, s.k, w.w13,
                                                  b["perm"], b["topk_w"], b["block_map"], b["num_blocks"], bn,
                                                  b["h"])),
                 ("gemm_tc_kernel down",
                  lambda: _lib.moe_expert_gemm_w4(_lib.DOWN, _lib.IMPL_TC, b["h"], T, s.H, s.F, s.E, s.k, w.w2,
                                                  b["perm"], b["topk_w"], b["block_map"], b["num_blocks"], bn,
                                                  b["y"]))]
    ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    words = np.zeros(_lib.moe_trace_words(), np.uint64)
    report = {"workload": a.workload, "block_n": bn, "ctas": ctas, "kernels": {}}
    for name, call in calls:
        call()  # warm: the first launch of a kernel pays for loading it
        torch.cuda.synchronize()
        _lib.moe_trace_reset()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        call()
        ev1.record()
        torch.cuda.synchronize()
        if _lib.moe_get_device_error():
            raise RuntimeError(f"{name}: the kernel reported a device error")
        _lib.moe_trace_read(words)
        report["kernels"][name] = {"us": ev0.elapsed_time(ev1) * 1e3, "roles": role_stats(words, ctas)}

    if a.json:
        print(json.dumps(report))
        return 0
    print(f"{a.workload}, block_n {bn}: share of each role's span spent in bounded mbarrier waits "
          f"(median over the CTAs [min, max]); the rest is the role's own work")
    for name, k in report["kernels"].items():
        print(f"\n{name}: {k['us']:.1f} us (one traced launch)")
        for role, r in k["roles"].items():
            print(f"  {role:17s} x{r['warps']:<2d} waits {r['wait_share_median']:.3f} "
                  f"[{r['wait_share_min']:.3f}, {r['wait_share_max']:.3f}]  waits/warp {r['waits_per_warp']:.0f}  "
                  f"span kcycles {r['span_kcycles_min']:.0f}-{r['span_kcycles_max']:.0f}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
