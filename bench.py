#!/usr/bin/env python3
"""Benchmark of the W4 MoE FFN layer forward (routing + grouped GEMMs + combine).

One step = one pass of the whole hot path over one batch of synthetic tokens:
moe_route -> gate/up GEMM (+SwiGLU) -> down GEMM -> moe_combine (at decode
sizes the fused decode kernel runs all four in one launch).  The default
workload is the 512-token prefill through the full-width layer (H=2048, 256
experts top-8 + 1 shared, F=512).  Weights (455 MB packed) exceed the 126 MB
L2, so every step streams them from HBM; decode workloads flush L2 between
steps instead.  The timed steps replay a CUDA graph of the layer call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill512|prefill4k|decode1|decode8|skew16k|tiny] [--only]
                  [--kernels auto|tc|gemv] [--block-n B] [--no-cpu-baseline]
                  [--no-e2e] [--no-graph]

The JSON line's top-level value is the chosen workload (default prefill512);
unless --only is given, the other workloads of the metric (4K-token prefill,
batch-1 and 8-token decode, the skewed 16K-token prefill) are timed the same
way in the same run and reported under "workloads", each with its roofline.
Under torchrun each rank runs the same workloads on its own GPU with its own
tokens (weak scaling, no collective on the data path); rank 0 prints one JSON
line.  `--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s (W4 routing+grouped GEMM) at T=512/4096; % of roofline"
L2_BYTES = 126 * 1024 * 1024


# --------------------------------------------------------------------------- #
# algorithmic work (per launch / per step)
# --------------------------------------------------------------------------- #
def expert_bytes(shape):
    """Packed uint4 weights + bf16 scale + bf16 bias of one expert's gate/up and down matrices."""
    H, F = shape.H, shape.F
    w13 = 2 * F * H // 2 + 2 * (2 * F * H // 64) * 2
    w2 = H * F // 2 + 2 * (H * F // 64) * 2
    return w13, w2


def algorithmic(shape, T, n_touched):
    w13, w2 = expert_bytes(shape)
    H, F, k, E = shape.H, shape.F, shape.k, shape.E
    A = T * k
    rows = A + T
    n = n_touched + 1
    gate_up_bytes = n * w13 + T * H * 2 + rows * F * 2            # weights + x + h
    down_bytes = n * w2 + rows * F * 2 + rows * H * 2              # weights + h + y
    ffn_bytes = n * (w13 + w2) + T * H * 2 + rows * H * 2          # both projections, h on chip: weights + x + y
    flops_gate_up = 2.0 * rows * 2 * F * H
    flops_down = 2.0 * rows * H * F
    step_bytes = n * (w13 + w2) + T * H * 2 + T * E * 4 + T * H * 2
    return {"gate_up_bytes": gate_up_bytes, "down_bytes": down_bytes, "ffn_bytes": ffn_bytes,
            "flops_gate_up": flops_gate_up,
            "flops_down": flops_down, "step_bytes": step_bytes, "step_flops": flops_gate_up + flops_down}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value across ranks (the timed region ends when the slowest rank ends)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_tokens(shape, T, rank, skew=False):
    """Each rank's own batch of T tokens (weak scaling: a distinct seed per rank)."""
    return workloads.make_tokens(shape, T, seed=rank, skew=skew)


# --------------------------------------------------------------------------- #
# clocks
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if not self.proc:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln.strip() for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append({"sm": float(p[1]), "max": float(p[2]), "power": float(p[3]) if p[3] not in
                             ("[N/A]", "N/A") else 0.0, "hw": p[5], "hwt": p[6], "swt": p[7], "pcap": p[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [r for r in rows if r["power"] > 300] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in busy])), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy)}


# --------------------------------------------------------------------------- #
# our implementation
# --------------------------------------------------------------------------- #
EXTRA_WORKLOADS = ("prefill4k", "decode1", "decode8", "skew16k")


def tensor_bound(T):
    """Above ~2K tokens the gate/up GEMM does enough FLOP per weight byte to be tensor-core bound."""
    return T >= 2048


def measure_workload(args, wl, layer, d, rank, world, dev):
    """Warm-up, a per-stage breakdown (eager launches with events), then the timed region: K replays of
    the layer step captured once as a CUDA graph (L2 flushed between steps when the step's bytes fit in
    L2), and the end-to-end number through moe_layer_forward_host.  Returns the workload's result."""
    import torch

    from bit_mixture_experts_gb300 import _lib

    s = wl.shape
    T = wl.T
    tok = rank_tokens(s, T, rank, wl.skew) if rank else d
    x = torch.from_numpy(tok["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(tok["logits"]).to(dev)
    out = torch.empty((T, s.H), dtype=torch.bfloat16, device=dev)
    b = layer.buffers(T)
    stream = torch.cuda.current_stream()
    impl, bn = layer.impl_for(T), layer.block_n_for(T)
    w = layer.weights
    fused_combine = impl == _lib.IMPL_TC and b.get("combine_ws") is not None
    fused_ffn = layer.h_on_chip(T)  # the layer runs both projections in one launch (moe_expert_ffn_w4)
    nseg = 3 if (fused_combine or fused_ffn) else 4

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        _lib.moe_route(logits, s.k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                       b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
        if ev is not None:
            ev[1].record(stream)
        if fused_ffn:
            # the layer's own path at these tile heights: both projections in one launch, h on chip
            _lib.moe_expert_ffn_w4(x, T, s.H, s.F, s.E, s.k, w.w13, w.w2, b["perm"], b["block_map"],
                                   b["num_blocks"], bn, b["y"])
            if ev is not None:
                ev[2].record(stream)
            _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], out)
            if ev is not None:
                ev[3].record(stream)
            return
        _lib.moe_expert_gemm_w4(_lib.GATE_UP, impl, x, T, s.H, s.F, s.E, s.k, w.w13, b["perm"], b["topk_w"],
                                b["block_map"], b["num_blocks"], bn, b["h"])
        if ev is not None:
            ev[2].record(stream)
        if fused_combine:
            # the layer's own path with the tensor-core kernel: the combine in the down GEMM's epilogue
            _lib.moe_down_combine(b["h"], T, s.H, s.F, s.E, s.k, w.w2, b["perm"], b["inv_perm"], b["topk_w"],
                                  b["block_map"], b["num_blocks"], bn, b["y"], out, b["combine_ws"])
            if ev is not None:
                ev[3].record(stream)
            return
        _lib.moe_expert_gemm_w4(_lib.DOWN, impl, b["h"], T, s.H, s.F, s.E, s.k, w.w2, b["perm"], b["topk_w"],
                                b["block_map"], b["num_blocks"], bn, b["y"])
        if ev is not None:
            ev[3].record(stream)
        _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], out)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    touched = int((b["counts"] > 0).sum().item())
    work = algorithmic(s, T, touched)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if work["step_bytes"] < 2 * L2_BYTES \
        else None

    def hold_stream():
        # Hold the stream busy for a moment so the host can queue the steps ahead of the GPU: at
        # decode sizes one host-side launch takes longer than the kernel, and the events would
        # otherwise time the host.  (The end-to-end number below keeps the host in its clock.)
        torch.cuda._sleep(int(min(100e-3, 0.3e-3 * args.steps + 2e-3) * 2.0e9))

    # per-stage breakdown: eager launches with events between the stages (not the timed region)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    hold_stream()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        step(events[i])
    torch.cuda.synchronize()
    seg = np.array([[events[i][j].elapsed_time(events[i][j + 1]) for j in range(nseg)] for i in range(args.steps)])
    assert _lib.moe_get_device_error() == 0, "device error word set"

    # the step captured once as a CUDA graph (the library launches only on the given stream and never
    # synchronises, so the whole layer is capturable); the timed region replays it
    graph, per_step_launches = None, None
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            n_cap = _lib.moe_launch_count()
            with torch.cuda.graph(g):
                # the layer's public entry point (moe_layer_forward): at decode sizes with the GEMV
                # kernel this is the fused single-launch decode kernel
                layer.forward(x, logits, out)
            per_step_launches = _lib.moe_launch_count() - n_cap
            g.replay()
            torch.cuda.synchronize()
            graph = g
        except Exception as ex:  # report the eager timing instead
            print(f"CUDA graph capture unavailable ({type(ex).__name__}: {ex}); timing eager launches",
                  file=sys.stderr)
            graph = None
            torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    time.sleep(0.1)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = _lib.moe_launch_count()
    hold_stream()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            layer.forward(x, logits, out)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    launches = (_lib.moe_launch_count() - n0) if graph is None else per_step_launches * args.steps
    if world > 1:
        torch.distributed.barrier()
    ms = float(np.mean([a.elapsed_time(b_) for a, b_ in ev]))
    ms = max_over_ranks(ms, world, dev)
    assert _lib.moe_get_device_error() == 0, "device error word set"

    # end to end through the C ABI with host buffers (pinned): x to the device, logits and out across
    # the host link inside the kernels, and a stream synchronisation in each step's wall-clock window;
    # the L2 flush between steps runs (and is waited for) outside the window
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(tok["x_bits"].view(np.int16)).pin_memory()
        lh = torch.from_numpy(tok["logits"]).pin_memory()
        oh = torch.empty((T, s.H), dtype=torch.int16).pin_memory()
        stage = {"x": torch.empty_like(x), "logits": torch.empty_like(logits), "out": torch.empty_like(out)}
        for _ in range(max(1, args.warmup)):
            layer.forward_host(xh, lh, oh, stage)
        torch.cuda.synchronize()
        ne = max(3, min(args.steps, 50))
        tot = 0.0
        for _ in range(ne):
            if flush is not None:
                flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            layer.forward_host(xh, lh, oh, stage)
            torch.cuda.synchronize()
            tot += time.perf_counter() - t0
        e2e_ms = tot * 1e3 / ne
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(xh.numel() * 2 + lh.numel() * 4),
               "d2h_bytes_per_step": int(oh.numel() * 2), "ms_per_step": e2e_ms,
               "note": "wall clock per step through moe_layer_forward_host with pinned host buffers: x copied to "
                       "the device, logits read by the routing kernel and out written by the combine (or the fused "
                       "decode kernel) over the host link, stream sync"}

    # roofline of the dominant kernel: the gate/up GEMM (the fused FFN kernel where the layer keeps h on
    # chip, the fused decode kernel at decode sizes)
    gu_ms = float(seg[:, 1].mean())
    peaks = load_peaks()
    fused_decode = impl == _lib.IMPL_GEMV and T <= 8
    if fused_decode:
        # one kernel is the whole step: its bytes (weights of the touched experts, x, logits, out)
        # over the step time
        achieved = work["step_bytes"] / (ms * 1e-3) / 1e9
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
    elif fused_ffn and not tensor_bound(T):
        achieved = work["ffn_bytes"] / (gu_ms * 1e-3) / 1e9
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
    elif fused_ffn:
        achieved = work["step_flops"] / (gu_ms * 1e-3) / 1e12
        peak, unit, bound = peaks["bf16_tflops"], "TFLOP/s", "tensor"
    elif tensor_bound(T):
        achieved = work["flops_gate_up"] / (gu_ms * 1e-3) / 1e12
        peak, unit, bound = peaks["bf16_tflops"], "TFLOP/s", "tensor"
    else:
        achieved = work["gate_up_bytes"] / (gu_ms * 1e-3) / 1e9
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
    kname = {_lib.IMPL_TC: "gemm_tc_kernel<0>", _lib.IMPL_TC2: "gemm_pair_kernel<0>",
             _lib.IMPL_GEMV: "gemv_kernel<0>"}.get(impl, str(impl))
    traffic = (profiled_traffic(wl.name, 0, kernel="ffn_tc_kernel") if fused_ffn else
               profiled_traffic(wl.name, 0) if impl == _lib.IMPL_TC else
               profiled_traffic(wl.name, 0, kernel="decode_kernel") if fused_decode else None)
    kdesc = ("decode_kernel: the fused layer (routing, gate/up, down and combine in one launch)" if fused_decode
             else "ffn_tc_kernel: both projections of every expert tile, h kept on chip (moe_expert_ffn_w4)"
             if fused_ffn else f"gate/up grouped GEMM {kname} (moe_expert_gemm_w4, MOE_GATE_UP_SWIGLU)")
    roof = {"kernel": kdesc, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": peaks["source"], "traffic": traffic,
            "algorithmic_per_launch": (work["step_bytes"] if fused_decode else
                                       (work["step_flops"] if tensor_bound(T) else work["ffn_bytes"]) if fused_ffn
                                       else work["flops_gate_up"] if tensor_bound(T) else work["gate_up_bytes"]),
            "launch_ms": ms if fused_decode else gu_ms}
    layer_tflops = work["step_flops"] / (ms * 1e-3) / 1e12
    layer_gbs = work["step_bytes"] / (ms * 1e-3) / 1e9
    return {
        "workload": wl.name, "desc": wl.desc, "T": T, "value": world * T / (ms * 1e-3), "unit": "tokens/s",
        "ms_per_step": ms, "steps": args.steps, "block_n": bn, "touched_experts": touched,
        "l2": ("L2 flushed between steps" if flush is not None else
               f"inputs larger than L2 ({work['step_bytes'] / 1e6:.0f} MB streamed per step)"),
        "stages_note": ("eager launches of the four entry points (moe_route, gate/up and down moe_expert_gemm_w4, "
                        "moe_combine); the timed step is the fused decode kernel") if fused_decode else
                       ("eager launches of the three entry points (moe_route, gate/up moe_expert_gemm_w4, "
                        "moe_down_combine); the timed step replays the same launches") if fused_combine else
                       ("eager launches of the three entry points the layer uses at these tile heights (moe_route, "
                        "moe_expert_ffn_w4, moe_combine); the timed step replays the same launches") if fused_ffn else
                       "eager launches of the four entry points; the timed step replays the same launches",
        "stages_ms": ({"route": float(seg[:, 0].mean()), "gate_up": gu_ms, "down_combine": float(seg[:, 2].mean())}
                      if fused_combine else
                      {"route": float(seg[:, 0].mean()), "ffn": gu_ms, "combine": float(seg[:, 2].mean())}
                      if fused_ffn else
                      {"route": float(seg[:, 0].mean()), "gate_up": gu_ms, "down": float(seg[:, 2].mean()),
                       "combine": float(seg[:, 3].mean())}),
        "roofline": roof,
        "layer_roofline": {"tflops": layer_tflops, "frac_bf16": layer_tflops / peaks["bf16_tflops"],
                           "hbm_gbs": layer_gbs, "frac_hbm": layer_gbs / peaks["hbm_gbs"],
                           "note": "whole step: 56.6 MFLOP per token, bytes of the touched experts + x, logits, out"},
        "gpu_launches": int(launches), "launch": "cuda_graph" if graph is not None else "eager",
        "e2e": e2e,
    }


def measure_host_synced(args, wl, layer, d, dev):
    """Ablation of GPU-resident routing (the pages credit it with +89% prefill): each step routes on the
    GPU, copies the per-expert counts to the host and waits for them, builds the block map on the host,
    copies it back, and launches one gate/up and one down GEMM per expert (the shared expert last), then
    the combine.  Same kernels and results; only the dispatch differs.  Wall clock per step."""
    import torch

    from bit_mixture_experts_gb300 import _lib

    s = wl.shape
    T = wl.T
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    out = torch.empty((T, s.H), dtype=torch.bfloat16, device=dev)
    b = layer.buffers(T)
    impl, bn = layer.impl_for(T), layer.block_n_for(T)
    w = layer.weights
    A = T * s.k
    counts_h = torch.empty(s.E, dtype=torch.int32).pin_memory()
    # per expert: its tile count 16 bytes apart and its block-map rows from a 16-byte boundary (4 rows),
    # as the library requires of every pointer
    nb_dev = torch.empty(4 * (s.E + 1), dtype=torch.int32, device=dev)
    bm_dev = torch.empty((_lib.moe_block_map_capacity(T, s.E, s.k, bn) + 4 * (s.E + 1), 3), dtype=torch.int32,
                         device=dev)

    def step():
        _lib.moe_route(logits, s.k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                       b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
        counts_h.copy_(b["counts"])
        torch.cuda.current_stream().synchronize()       # the host waits for the routing
        c = counts_h.numpy()
        rows, first, nbs, off = [], [], [], 0
        for e in range(s.E + 1):
            n = int(c[e]) if e < s.E else T
            r0 = off if e < s.E else A
            rows += [(0, 0, 0)] * (-len(rows) % 4)
            first.append(len(rows))
            rows += [(e, r0 + i, min(bn, n - i)) for i in range(0, n, bn)]
            nbs.append(len(rows) - first[-1])
            off += n if e < s.E else 0
        bm_dev[:len(rows)].copy_(torch.tensor(rows, dtype=torch.int32))
        nb_dev.copy_(torch.tensor([[v, 0, 0, 0] for v in nbs], dtype=torch.int32).view(-1))
        launches = 2
        for mode, act, wt, dst in ((_lib.GATE_UP, x, w.w13, b["h"]), (_lib.DOWN, b["h"], w.w2, b["y"])):
            for e in range(s.E + 1):
                if nbs[e] == 0:
                    continue
                _lib.moe_expert_gemm_w4(mode, impl, act, T, s.H, s.F, s.E, s.k, wt, b["perm"], b["topk_w"],
                                        bm_dev.data_ptr() + 12 * first[e], nb_dev.data_ptr() + 16 * e, bn, dst)
                launches += 1
        _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], out)
        return launches

    for _ in range(max(2, args.warmup)):
        launches = step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / n
    assert _lib.moe_get_device_error() == 0, "device error word set"
    fused = layer.forward(x, logits)  # the same layer through its single-stream path
    torch.cuda.synchronize()
    same = bool(torch.equal(fused.view(torch.int16), out.view(torch.int16)))
    return {"ms_per_step": ms, "value": T / (ms * 1e-3), "unit": "tokens/s", "steps": n, "same_output": same,
            "launches_per_step": launches,
            "note": "routing on the GPU, counts to the host (synchronised), block map built on the host, one "
                    "GEMM launch per expert and projection; wall clock per step"}


def measure_chain(args, dev, T=1, L=4):
    """Decode through L layers in sequence (layer.MoEDecodeChain): each layer's logits are the router
    projection of the previous layer's output, then the fused decode kernel; 2 L launches per step,
    replayed as one CUDA graph, L2 flushed between steps.  Reports the time per layer and, per layer,
    the bytes of its touched experts' weights and its router matrix against the HBM roofline."""
    import torch

    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoEDecodeChain

    s = workloads.FULL
    ws = [workloads.make_weights(s, seed=100 + l) for l in range(L)]
    wrs = [workloads.router_weight_bits(s, seed=100 + l) for l in range(L)]
    chain = MoEDecodeChain(s.H, s.E, s.k, s.F, ws, wrs, device=dev, impl="gemv")
    del ws
    tok = workloads.make_tokens(s, T, seed=7)
    x = torch.from_numpy(tok["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    for _ in range(max(3, args.warmup)):
        chain.forward(x)
    torch.cuda.synchronize()
    touched = [int((layer.buffers(T)["counts"] > 0).sum().item()) for layer in chain.layers]
    g = torch.cuda.CUDAGraph()
    n_cap = _lib.moe_launch_count()
    with torch.cuda.graph(g):
        chain.forward(x)
    launches = _lib.moe_launch_count() - n_cap
    g.replay()
    torch.cuda.synchronize()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda._sleep(int(min(100e-3, 0.3e-3 * args.steps + 2e-3) * 2.0e9))
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0, "device error word set"
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    w13, w2 = expert_bytes(s)
    # per layer: the touched experts' weights, the router matrix, and x / its norm / out / logits
    step_bytes = sum((n + 1) * (w13 + w2) for n in touched) + L * (s.E * s.H * 2 + 3 * T * s.H * 2 + T * s.E * 4)
    peaks = load_peaks()
    gbs = step_bytes / (ms * 1e-3) / 1e9
    return {"layers": L, "T": T, "ms_per_step": ms, "us_per_layer": 1e3 * ms / L, "value": T * L / (ms * 1e-3),
            "unit": "layer-tokens/s", "gpu_launches_per_step": int(launches), "touched_experts": touched,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "algorithmic_per_step": int(step_bytes),
                         "note": "per layer: touched experts' W4 weights + the bf16 router matrix + x, logits, out"},
            "note": "each layer: RMS norm of the previous layer's output and its router logits (moe_norm_router, "
                    "one launch), then the fused decode kernel; one CUDA graph per step, L2 flushed between steps"}


def measure_unfused(args, wl, d, dev, fused_ms):
    """Ablation of the fused dequantisation (the pages credit it with +77.4% prefill): the same layer
    with the weights first expanded to a bf16 copy in HBM (moe_expand_w4), then the same tensor-core
    kernel reading that copy (MOE_IMPL_TC_BF16).  Two timings: the expansion in every step (the
    dequantise-then-GEMM pipeline), and a resident bf16 copy (3.6 times the weight bytes per step, and
    1.6 GB of memory for this layer).  CUDA events on the stream, inputs larger than L2."""
    import torch

    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4

    s = wl.shape
    T = wl.T
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, device=dev, impl="tc_bf16", block_n=args.block_n)
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    out = torch.empty((T, s.H), dtype=torch.bfloat16, device=dev)
    p13, p2 = d["w13_packed"].shape, d["w2_packed"].shape

    def timed(expand):
        for _ in range(max(2, args.warmup)):
            if expand:
                layer.expand(layer.w13_r, p13, layer.w13_x)
                layer.expand(layer.w2_r, p2, layer.w2_x)
            layer.forward(x, logits, out)
        torch.cuda.synchronize()
        n = max(3, min(args.steps, 20))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            if expand:
                layer.expand(layer.w13_r, p13, layer.w13_x)
                layer.expand(layer.w2_r, p2, layer.w2_x)
            layer.forward(x, logits, out)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    ms_expand = timed(True)
    ms_resident = timed(False)
    assert _lib.moe_get_device_error() == 0, "device error word set"
    bf16_bytes = layer.w13_x.numel() + layer.w2_x.numel()
    return {"expand_every_step_ms": ms_expand, "resident_bf16_copy_ms": ms_resident, "fused_ms_per_step": fused_ms,
            "fused_speedup_vs_expand": ms_expand / fused_ms, "fused_speedup_vs_resident": ms_resident / fused_ms,
            "bf16_copy_bytes": int(bf16_bytes),
            "note": "moe_expand_w4 (bf16 copy of all 257 experts' weights) then the tensor-core kernel on that "
                    "copy; same results bit for bit"}


def measure_fused_combine(args, wl, layer, d, dev):
    """Ablation of the combine's own launch: the step with the combine in the down GEMM's epilogue
    (moe_down_combine; same bits) against the step as the layer runs it (down GEMM, then moe_combine).
    CUDA events on the stream around each eager step, L2 flushed between steps."""
    import torch

    from bit_mixture_experts_gb300 import _lib

    s = wl.shape
    T = wl.T
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    out = torch.empty((T, s.H), dtype=torch.bfloat16, device=dev)
    ref = torch.empty_like(out)
    b = layer.buffers(T)
    impl, bn = layer.impl_for(T), layer.block_n_for(T)
    if impl != _lib.IMPL_TC:
        return None
    w = layer.weights
    ws = torch.zeros(_lib.moe_down_combine_workspace_size(T, s.H) // 4, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step(fused, o):
        _lib.moe_route(logits, s.k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                       b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
        _lib.moe_expert_gemm_w4(_lib.GATE_UP, impl, x, T, s.H, s.F, s.E, s.k, w.w13, b["perm"], b["topk_w"],
                                b["block_map"], b["num_blocks"], bn, b["h"])
        if fused:
            _lib.moe_down_combine(b["h"], T, s.H, s.F, s.E, s.k, w.w2, b["perm"], b["inv_perm"], b["topk_w"],
                                  b["block_map"], b["num_blocks"], bn, b["y"], o, ws)
        else:
            _lib.moe_expert_gemm_w4(_lib.DOWN, impl, b["h"], T, s.H, s.F, s.E, s.k, w.w2, b["perm"], b["topk_w"],
                                    b["block_map"], b["num_blocks"], bn, b["y"])
            _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], o)

    def timed(fused, o):
        for _ in range(max(3, args.warmup)):
            step(fused, o)
        n = max(3, min(args.steps, 30))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            flush.zero_()
            ev[i][0].record()
            step(fused, o)
            ev[i][1].record()
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b_) for a, b_ in ev]))

    ms_sep = timed(False, ref)
    ms_fused = timed(True, out)
    assert _lib.moe_get_device_error() == 0, "device error word set"
    return {"fused_combine_ms_per_step": ms_fused, "separate_combine_ms_per_step": ms_sep,
            "same_output": bool(torch.equal(out.view(torch.int16), ref.view(torch.int16))),
            "workspace_left_zero": int(ws.count_nonzero().item()) == 0,
            "note": "eager steps (route, gate/up, then moe_down_combine or down GEMM + moe_combine); the layer "
                    "keeps the separate combine, which measures faster"}


def measure_fused_ffn(args, wl, layer, d, dev):
    """Ablation of h kept on chip: the layer's step with both projections of each expert tile in one
    launch (moe_expert_ffn_w4) against the same step with the two grouped GEMMs and h through HBM (same
    bits).  CUDA events on the stream around each eager step, L2 flushed between steps.  Only where the
    layer keeps h on chip (tiles of at most 64 rows)."""
    import torch

    from bit_mixture_experts_gb300 import _lib

    s = wl.shape
    T = wl.T
    if not layer.h_on_chip(T):
        return None
    x = torch.from_numpy(d["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.from_numpy(d["logits"]).to(dev)
    outs = {n: torch.empty((T, s.H), dtype=torch.bfloat16, device=dev) for n in ("fused", "two")}
    b = layer.buffers(T)
    bn = layer.block_n_for(T)
    w = layer.weights
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step(fused, o):
        _lib.moe_route(logits, s.k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                       b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
        if fused:
            _lib.moe_expert_ffn_w4(x, T, s.H, s.F, s.E, s.k, w.w13, w.w2, b["perm"], b["block_map"],
                                   b["num_blocks"], bn, b["y"])
        else:
            _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_TC, x, T, s.H, s.F, s.E, s.k, w.w13, b["perm"],
                                    b["topk_w"], b["block_map"], b["num_blocks"], bn, b["h"])
            _lib.moe_expert_gemm_w4(_lib.DOWN, _lib.IMPL_TC, b["h"], T, s.H, s.F, s.E, s.k, w.w2, b["perm"],
                                    b["topk_w"], b["block_map"], b["num_blocks"], bn, b["y"])
        _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], o)

    def timed(fused, o):
        for _ in range(max(3, args.warmup)):
            step(fused, o)
        n = max(3, min(args.steps, 30))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            flush.zero_()
            ev[i][0].record()
            step(fused, o)
            ev[i][1].record()
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b_) for a, b_ in ev]))

    ms_two = timed(False, outs["two"])
    ms_fused = timed(True, outs["fused"])
    assert _lib.moe_get_device_error() == 0, "device error word set"
    return {"fused_ffn_ms_per_step": ms_fused, "two_gemms_ms_per_step": ms_two,
            "same_output": bool(torch.equal(outs["fused"].view(torch.int16), outs["two"].view(torch.int16))),
            "note": "eager steps: route, then moe_expert_ffn_w4 (the layer's path here) or the gate/up and down "
                    "grouped GEMMs with h through HBM, then moe_combine"}


def run_ours(args, rank, world, local_rank):
    import torch

    from bit_mixture_experts_gb300 import build
    from bit_mixture_experts_gb300.layer import MoELayerW4

    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    names = [args.workload] + ([] if args.only else [n for n in EXTRA_WORKLOADS if n != args.workload])
    layers = {}
    results = {}
    clocks = ClockSampler(local_rank) if rank == 0 else None
    primary_d = None
    for name in names:
        wl = workloads.WORKLOADS[name]
        s = wl.shape
        d = workloads.make_workload(wl, seed=0, with_weights=s not in layers)
        if s not in layers:
            layers[s] = (MoELayerW4(s.H, s.E, s.k, s.F, d, device=dev, impl=args.kernels, block_n=args.block_n), d)
        layer, wd = layers[s]
        d.update({n_: v for n_, v in wd.items() if n_.startswith(("w13_", "w2_"))})
        if name == args.workload:
            primary_d = d
        results[name] = measure_workload(args, wl, layer, d, rank, world, dev)
    if not args.only and rank == 0 and world == 1:
        results["decode1_chain4"] = measure_chain(args, dev, T=1, L=4)
    ablations = {}
    if not args.no_ablations and rank == 0 and world == 1 and args.workload in ("prefill512", "prefill4k"):
        wl = workloads.WORKLOADS[args.workload]
        layer, wd = layers[wl.shape]
        hs = measure_host_synced(args, wl, layer, primary_d, dev)
        hs["fused_ms_per_step"] = results[args.workload]["ms_per_step"]
        hs["fused_speedup"] = hs["ms_per_step"] / results[args.workload]["ms_per_step"]
        ablations["host_synced_routing"] = hs
        ablations["fused_combine"] = measure_fused_combine(args, wl, layer, primary_d, dev)
        ablations["fused_ffn"] = measure_fused_ffn(args, wl, layer, primary_d, dev)
        ablations["unfused_dequant"] = measure_unfused(args, wl, primary_d, dev, results[args.workload]["ms_per_step"])
    if clocks:
        clocks.stop()
    p = results[args.workload]
    wl = workloads.WORKLOADS[args.workload]
    s = wl.shape
    res = {
        "metric": METRIC, "value": p["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": p["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x uint4 (fp32 accumulate)",
        "data": "synthetic (seeded; random-init uint4 weights, bf16 scales/biases)",
        "config": {"workload": wl.name, "desc": wl.desc, "T": wl.T, "H": s.H, "E": s.E, "k": s.k, "F": s.F,
                   "shared_experts": 1, "group": 64, "block_n": p["block_n"], "kernels": args.kernels,
                   "touched_experts": p["touched_experts"], "l2": p["l2"],
                   "parallelism": f"replicas x{world} (tokens sharded, no collective)"},
        "stages_note": p["stages_note"], "stages_ms": p["stages_ms"],
        "roofline": p["roofline"], "layer_roofline": p["layer_roofline"],
        "gpu_launches": p["gpu_launches"], "launch": p["launch"], "e2e": p["e2e"],
        "workloads": {n: r for n, r in results.items() if n != args.workload},
        "ablations": ablations,
        "workloads_note": ("the other workloads of the metric, each timed the same way right after the primary "
                           "one (same clocks record); prefill4k and skew16k report the gate/up kernel against the "
                           "bf16 tensor peak, decode1/decode8 the fused decode kernel against HBM; decode1_chain4 "
                           "is batch-1 decode through four dependent layers (router projection + fused decode "
                           "kernel per layer)"),
    }
    if clocks:
        res["clocks"] = clocks.summary()
    return res, primary_d


KERNEL_SOURCES = {
    "gemm_tc_kernel": ("moe_gemm_tc.cu", "moe_tc_dev.cuh", "moe_tmap.cuh", "moe_ptx.cuh", "moe_common.cuh"),
    "decode_kernel": ("moe_decode.cu", "moe_gemv_dev.cuh", "moe_route_dev.cuh", "moe_ptx.cuh", "moe_common.cuh"),
    "ffn_tc_kernel": ("moe_ffn_tc.cu", "moe_tc_dev.cuh", "moe_ptx.cuh", "moe_common.cuh"),
}


def kernel_source_sha(kernel="gemm_tc_kernel"):
    """sha256[:16] of a kernel's source code with comments and blank space removed (the profile
    summaries record the one they measured, so an edit of comments alone keeps them valid)."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_mixture_experts_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        code = []
        for line in text.split("\n"):
            # drop a // comment unless the // sits inside a string literal on that line
            cut = line.find("//")
            if cut >= 0 and line[:cut].count('"') % 2 == 0:
                line = line[:cut]
            line = " ".join(line.split())
            if line:
                code.append(line)
        h.update("\n".join(code).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, mode, kernel="gemm_tc_kernel"):
    """DRAM bytes per launch of the kernel (gemm_tc_kernel<mode>, or decode_kernel with mode 0) from the
    committed ncu summary of this workload, or None when there is none or the kernel's sources changed
    since it was taken."""
    p = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.md")
    if not os.path.exists(p):
        return None
    sha, traffic = None, None
    with open(p) as f:
        for line in f:
            if line.startswith("kernel source sha256"):
                sha = line.rsplit("`", 2)[-2]
            if line.startswith(f"traffic_bytes_per_launch mode{mode}:"):
                traffic = int(line.split(":")[1])
    return traffic if sha == kernel_source_sha(kernel) else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------- #
# CPU oracle (reference arm and cpu_baseline)
# --------------------------------------------------------------------------- #
def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def time_oracle(d, n_tokens, budget_s=20.0):
    """Time the float64 oracle on the first n_tokens of the workload (all their experts)."""
    from oracle import moe_ref
    wl = d["workload"]
    T = wl.T
    n = min(T, n_tokens)
    toks = np.arange(n)
    t0 = time.perf_counter()
    moe_ref.moe_forward(d["x_bits"], d["logits"], d, wl.shape.k, tokens=toks)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle_cores(), "kind": "oracle",
            "sample": f"first {n} of the {T} tokens of {wl.name}, all their routed experts + the shared expert "
                      f"dequantised and multiplied in float64 NumPy ({dt:.1f} s)", "seconds": dt}


ONE_CORE_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def time_oracle_one_core(workload, n_tokens):
    """The same oracle sample in a fresh interpreter whose BLAS is limited to one thread (the
    thread count is fixed when NumPy loads its BLAS, so it cannot be lowered in this process)."""
    code = ("import json, sys; sys.path.insert(0, %r); import bench, workloads; "
            "d = workloads.make_workload(%r, 0); print(json.dumps(bench.time_oracle(d, %d)))"
            % (ROOT, workload, n_tokens))
    env = dict(os.environ)
    env.update(ONE_CORE_ENV)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    res["cores"] = 1
    return res


def cpu_baseline(d):
    """The oracle on a bounded sample of the workload, with all host cores (BLAS threads) and with one."""
    wl = d["workload"]
    n = oracle_sample_tokens(wl)
    allc = time_oracle(d, n)
    one = time_oracle_one_core(wl.name, n)
    allc["one_core"] = one
    return allc


def oracle_sample_tokens(wl):
    return {"tiny": 64, "decode1": 1, "decode8": 8, "prefill512": 64, "prefill4k": 64, "skew16k": 64}[wl.name]


def run_reference(args):
    wl = workloads.WORKLOADS[args.workload]
    d = workloads.make_workload(wl, seed=0)
    n = oracle_sample_tokens(wl)
    # warm-up: W untimed runs of the same code on one token each (imports, BLAS threads, caches)
    for _ in range(max(0, args.warmup)):
        time_oracle(d, 1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(max(1, args.steps)):   # each step one bounded sample; stop after ~90 s of CPU work
        vals.append(time_oracle(d, n))
        if time.perf_counter() - t0 > 90.0:
            break
    wall = time.perf_counter() - t0
    v = float(np.median([x["value"] for x in vals]))
    cb = dict(vals[0])
    cb["value"] = v
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": len(vals), "warmup": max(0, args.warmup), "ms_per_step": 1e3 * n / v, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "desc": wl.desc, "T": wl.T, "sample_tokens": n},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill512", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--kernels", default="auto", choices=["auto", "tc", "tc2", "gemv"])
    ap.add_argument("--only", action="store_true", help="time the chosen workload alone (no per-workload extras)")
    ap.add_argument("--block-n", type=int, default=None, help="rows per GEMM tile (default: per kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a captured CUDA graph")
    ap.add_argument("--no-ablations", action="store_true", help="skip the ablation measurements")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res, d = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(d)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
