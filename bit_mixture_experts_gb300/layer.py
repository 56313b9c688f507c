"""A W4 mixture-of-experts FFN layer driven through the C ABI.

PyTorch only provides device memory and the stream; every step (routing,
grouped GEMMs, combine) runs in libmoe_w4.so's kernels.
"""
from __future__ import annotations

import numpy as np

from . import _lib

DEFAULT_BLOCK_N = {_lib.IMPL_TC: 128, _lib.IMPL_GEMV: 8, _lib.IMPL_TC2: 128, _lib.IMPL_TC_BF16: 128}
DECODE_MAX_T = 16  # token counts up to this take the GEMV kernel under impl="auto"


def default_block_n(impl: int, T: int, E: int, k: int) -> int:
    """Tile height of the block map for T tokens.

    The tensor-core kernel expands a 256-row slice of an expert's weights once
    per tile, so tiles should be as tall as the expert's rows allow: with fewer
    than 64 assignments per expert on average (512-token prompts through 256
    experts top-8 average 16) 64-row tiles waste less of the MMA on padding and
    give the grid more tiles; from there on 128-row tiles halve the
    dequantisation per token.  The GEMV kernel takes tiles of up to 8 rows.
    """
    if impl in (_lib.IMPL_TC, _lib.IMPL_TC2, _lib.IMPL_TC_BF16) and T * k < 64 * E:
        return 64
    return DEFAULT_BLOCK_N[impl]


def _dev(a: np.ndarray, device):
    """numpy -> torch on `device` keeping the bits (uint32 as int32, uint16 as int16)."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class MoELayerW4:
    """One layer: E routed experts (top-k) + 1 shared expert, hidden H, expert width F.

    `weights` holds the canonical arrays of the workloads module (w13_packed,
    w13_scale, w13_bias, w2_packed, w2_scale, w2_bias) as numpy arrays or torch
    tensors already on the device.
    """

    def __init__(self, H, E, k, F, weights: dict, device="cuda", impl="auto", block_n=None, fuse_combine=False):
        import torch
        self.H, self.E, self.k, self.F = H, E, k, F
        self.device = torch.device(device)
        self.impl = _lib.IMPLS[impl] if isinstance(impl, str) else int(impl)
        if H % 128 or F % 128:
            raise ValueError(f"H={H} and F={F} must be multiples of 128 (the kernels' K and M steps)")
        self.block_n = block_n  # None: chosen per token count by default_block_n
        # tensor-core path: the combine in the down GEMM's epilogue (moe_down_combine) instead of its own
        # launch; off by default, as it measures slower: the epilogue's counts, fences and gathers lengthen
        # every unit's epilogue beyond the next unit's main loop
        self.fuse_combine = fuse_combine
        _lib.load()
        w = {n: (v if isinstance(v, torch.Tensor) else _dev(v, self.device)) for n, v in weights.items()
             if n.startswith(("w13_", "w2_"))}
        # the CTA-pair kernel reads interleaved gate/up tiles, every other kernel the paired ones
        self.w13_r = self._repack(w["w13_packed"], w["w13_scale"], w["w13_bias"],
                                  gate_up=2 if self.impl == _lib.IMPL_TC2 else 1)
        self.w2_r = self._repack(w["w2_packed"], w["w2_scale"], w["w2_bias"], gate_up=False)
        if self.impl == _lib.IMPL_TC_BF16:
            # the unfused comparison path: a resident bf16 copy of the expanded weights
            self.w13_x = self.expand(self.w13_r, w["w13_packed"].shape)
            self.w2_x = self.expand(self.w2_r, w["w2_packed"].shape)
            self.weights = _lib.Weights(self.w13_x.data_ptr(), self.w2_x.data_ptr())
        else:
            self.weights = _lib.Weights(self.w13_r.data_ptr(), self.w2_r.data_ptr())
        self._bufs = {}

    def _repack(self, packed, scale, bias, gate_up):
        import torch
        n_mat, rows, kw = packed.shape
        nbytes = _lib.moe_repacked_bytes(n_mat, rows, kw * 8)
        out = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        _lib.moe_repack_w4(packed, scale, bias, gate_up, out)
        return out

    def expand(self, repacked, packed_shape, out=None):
        """bf16 copy of repacked weights (moe_expand_w4) for packed canonical shape [n_mat, rows, K/8]."""
        import torch
        n_mat, rows, kw = packed_shape
        if out is None:
            out = torch.empty(_lib.moe_expanded_bytes(n_mat, rows, kw * 8), dtype=torch.uint8, device=self.device)
        _lib.moe_expand_w4(repacked, n_mat, rows, kw * 8, out)
        return out

    def h_on_chip(self, T):
        """Whether the layer call for T tokens runs both projections as moe_expert_ffn_w4 (h kept in shared
        memory, the h buffer not written): the tensor-core kernel with tiles of at most 64 rows and
        F % 256 == 0, as moe_layer_forward decides."""
        return (self.impl_for(T) == _lib.IMPL_TC and self.block_n_for(T) <= 64 and self.F % 256 == 0
                and self.H % 128 == 0 and not self.fuse_combine)

    def impl_for(self, T):
        """GEMM kernel used for T tokens: under "auto", GEMV for decode-sized T, else tensor cores."""
        if self.impl != _lib.IMPL_AUTO:
            return self.impl
        return _lib.IMPL_GEMV if T <= DECODE_MAX_T and (self.block_n or 8) <= 8 else _lib.IMPL_TC

    def block_n_for(self, T):
        """Block-map tile height used for T tokens."""
        return self.block_n or default_block_n(self.impl_for(T), T, self.E, self.k)

    def buffers(self, T):
        """Routing / intermediate buffers for T tokens (allocated once per T)."""
        import torch
        if T in self._bufs:
            return self._bufs[T]
        E, k, H, F, bn = self.E, self.k, self.H, self.F, self.block_n_for(T)
        A = T * k
        dev = self.device
        cap = _lib.moe_block_map_capacity(T, E, k, bn)
        wsb = _lib.moe_route_workspace_size(T, E, k, bn)
        t = {
            "topk_ids": torch.empty((T, k), dtype=torch.int32, device=dev),
            "topk_w": torch.empty((T, k), dtype=torch.float32, device=dev),
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "perm": torch.empty(A, dtype=torch.int32, device=dev),
            "inv_perm": torch.empty(A, dtype=torch.int32, device=dev),
            "block_map": torch.empty((cap, 3), dtype=torch.int32, device=dev),
            "num_blocks": torch.empty(1, dtype=torch.int32, device=dev),
            "h": torch.empty((A + T, F), dtype=torch.bfloat16, device=dev),
            "y": torch.empty((A + T, H), dtype=torch.bfloat16, device=dev),
            "workspace": torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev),  # zero once, left zero
        }
        # counters of the fused decode kernel (used for T <= 8 with the GEMV kernel): zero once, left zero
        dws = _lib.moe_decode_workspace_size(T, H)
        t["decode_ws"] = torch.zeros(max(dws, 16), dtype=torch.uint8, device=dev) if dws else None
        # counters of the down GEMM's fused combine (tensor-core path): zero once, left zero
        cws = _lib.moe_down_combine_workspace_size(T, H) if self.fuse_combine else 0
        t["combine_ws"] = torch.zeros(max(cws, 16), dtype=torch.uint8, device=dev) if cws else None
        t["struct"] = _lib.Buffers(*(t[n].data_ptr() for n in ("topk_ids", "topk_w", "counts", "offsets", "perm",
                                                                 "inv_perm", "block_map", "num_blocks", "h", "y",
                                                                 "workspace")), wsb,
                                   t["decode_ws"].data_ptr() if dws else None, dws,
                                   t["combine_ws"].data_ptr() if cws else None, cws)
        self._bufs[T] = t
        return t

    def forward(self, x, logits, out=None, stream=None):
        """x bf16 [T, H], logits fp32 [T, E] on the device -> out bf16 [T, H]."""
        import torch
        T = x.shape[0]
        assert x.dtype == torch.bfloat16 and x.shape == (T, self.H) and x.is_contiguous()
        assert logits.dtype == torch.float32 and logits.shape == (T, self.E) and logits.is_contiguous()
        b = self.buffers(T)
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device)
        _lib.moe_layer_forward(x, logits, out, T, self.H, self.F, self.E, self.k, self.block_n_for(T),
                               self.impl_for(T), self.weights, b["struct"], stream)
        return out

    def forward_host(self, x_host, logits_host, out_host, stage, stream=None):
        """Host (pinned) x, logits, out; `stage` holds device x, logits, out of the same shapes."""
        T = x_host.shape[0]
        b = self.buffers(T)
        _lib.moe_layer_forward_host(x_host, logits_host, out_host, stage["x"], stage["logits"], stage["out"], T,
                                    self.H, self.F, self.E, self.k, self.block_n_for(T), self.impl_for(T), self.weights,
                                    b["struct"], stream)


class MoEDecodeChain:
    """Several MoE layers in sequence for small-batch decode (T <= 8 with the GEMV kernel): layer l's
    input is the RMS norm of layer l-1's output (of x for layer 0), and its router logits are its own
    router projection of that input, so the layers depend on each other as in a model's decode step.
    Two launches per layer: moe_norm_router (the norm and the logits), then moe_layer_forward (the
    fused decode kernel, which takes the top-k), all on one stream and capturable as one CUDA graph.

    `layer_weights` holds one canonical weight dict per layer (as MoELayerW4 takes), `router_bits` one
    bf16 router matrix [E, H] (uint16 bits) per layer.
    """

    def __init__(self, H, E, k, F, layer_weights, router_bits, device="cuda", impl="auto", block_n=None):
        import torch
        assert len(layer_weights) == len(router_bits) >= 1
        self.H, self.E, self.k, self.F = H, E, k, F
        self.device = torch.device(device)
        self.layers = [MoELayerW4(H, E, k, F, w, device=self.device, impl=impl, block_n=block_n)
                       for w in layer_weights]
        self.wr = [_dev(np.asarray(b, dtype=np.uint16), self.device) for b in router_bits]
        self._bufs = {}

    def buffers(self, T):
        """Per-layer outputs (bf16 [T, H]), logits (fp32 [T, E]) and the router's top-k scratch."""
        import torch
        if T not in self._bufs:
            dev, L = self.device, len(self.layers)
            self._bufs[T] = {
                "xn": [torch.empty((T, self.H), dtype=torch.bfloat16, device=dev) for _ in range(L)],
                "out": [torch.empty((T, self.H), dtype=torch.bfloat16, device=dev) for _ in range(L)],
                "logits": [torch.empty((T, self.E), dtype=torch.float32, device=dev) for _ in range(L)],
                "ids": [torch.empty((T, self.k), dtype=torch.int32, device=dev) for _ in range(L)],
                "w": [torch.empty((T, self.k), dtype=torch.float32, device=dev) for _ in range(L)],
            }
            for layer in self.layers:
                layer.buffers(T)
        return self._bufs[T]

    def forward(self, x, stream=None):
        """x bf16 [T, H] on the device -> the last layer's output (a buffer of the chain)."""
        T = x.shape[0]
        b = self.buffers(T)
        cur = x
        for l, layer in enumerate(self.layers):
            _lib.moe_norm_router(cur, self.wr[l], b["xn"][l], b["logits"][l], stream=stream)
            layer.forward(b["xn"][l], b["logits"][l], b["out"][l], stream)
            cur = b["out"][l]
        return cur
