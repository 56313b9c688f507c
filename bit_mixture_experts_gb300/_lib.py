"""ctypes binding of libmoe_w4.so: argument marshalling only.

Every function here takes torch tensors (or plain ints), checks dtypes and
shapes, passes raw pointers and the current CUDA stream to the C ABI of
include/moe_w4.h, and raises MoeError on a non-zero status.  No arithmetic of
the layer happens in Python; when the library is missing the import fails
loudly instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_w4.so")

MOE_OK = 0
ERRORS = {-1: "MOE_ERR_NULL", -2: "MOE_ERR_ALIGN", -3: "MOE_ERR_SHAPE", -4: "MOE_ERR_WORKSPACE",
          -5: "MOE_ERR_CUDA", -6: "MOE_ERR_DEVICE", -7: "MOE_ERR_MODE"}
DEVICE_ERRORS = {0: "ok", 1: "MOE_DEV_BAD_BLOCK", 2: "MOE_DEV_BAD_INDEX", 3: "MOE_DEV_TIMEOUT", 4: "MOE_DEV_BAD_WORKSPACE"}

GATE_UP, DOWN = 0, 1
IMPL_AUTO, IMPL_TC, IMPL_GEMV, IMPL_TC2, IMPL_TC_BF16 = 0, 2, 3, 4, 5
IMPLS = {"auto": IMPL_AUTO, "tc": IMPL_TC, "gemv": IMPL_GEMV, "tc2": IMPL_TC2, "tc_bf16": IMPL_TC_BF16}

# Exported symbols of include/moe_w4.h (checked by the CPU tests).
SYMBOLS = ["moe_version", "moe_launch_count", "moe_route_noalloc", "moe_route_x", "moe_router", "moe_rms_norm", "moe_norm_router",
           "moe_down_combine", "moe_down_combine_workspace_size", "moe_expert_ffn_w4", "moe_block_map_capacity", "moe_route_workspace_size", "moe_route",
           "moe_repacked_bytes", "moe_repack_w4", "moe_expanded_bytes", "moe_expand_w4", "moe_expert_gemm_w4", "moe_combine", "moe_decode_workspace_size",
           "moe_layer_forward", "moe_layer_forward_host", "moe_get_device_error", "moe_set_wait_limit_ns",
           "moe_trace_words", "moe_trace_reset", "moe_trace_read"]


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code} ({ERRORS.get(code, 'unknown')})")
        self.code = code


_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class Weights(ctypes.Structure):
    _fields_ = [("w13", _vp), ("w2", _vp)]


class Buffers(ctypes.Structure):
    _fields_ = [("topk_ids", _vp), ("topk_w", _vp), ("counts", _vp), ("offsets", _vp), ("perm", _vp),
                ("inv_perm", _vp), ("block_map", _vp), ("num_blocks", _vp), ("h", _vp), ("y", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("decode_ws", _vp), ("decode_ws_bytes", _sz),
                ("combine_ws", _vp), ("combine_ws_bytes", _sz)]


_SIGS = {
    "moe_version": ([], _i),
    "moe_launch_count": ([], ctypes.c_uint64),
    "moe_block_map_capacity": ([_i, _i, _i, _i], _i),
    "moe_route_workspace_size": ([_i, _i, _i, _i], _sz),
    "moe_route": ([_vp, _i, _i, _i, _i] + [_vp] * 9 + [_sz, _vp], _i),
    "moe_route_noalloc": ([_vp, _i, _i, _i, _i] + [_vp] * 9, _i),
    "moe_route_x": ([_vp, _vp, _i, _i, _i, _i, _i] + [_vp] * 10 + [_sz, _vp], _i),
    "moe_router": ([_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp], _i),
    "moe_rms_norm": ([_vp, _vp, _i, _i, ctypes.c_float, _vp], _i),
    "moe_norm_router": ([_vp, _vp, _i, _i, _i, ctypes.c_float, _vp, _vp, _vp], _i),
    "moe_down_combine_workspace_size": ([_i, _i], _sz),
    "moe_expert_ffn_w4": ([_vp, _i, _i, _i, _i, _i] + [_vp] * 5 + [_i, _vp, _vp], _i),
    "moe_down_combine": ([_vp, _i, _i, _i, _i, _i] + [_vp] * 6 + [_i, _vp, _vp, _vp, _sz, _vp], _i),
    "moe_repacked_bytes": ([_i, _i, _i], _sz),
    "moe_expanded_bytes": ([_i, _i, _i], _sz),
    "moe_expand_w4": ([_vp, _i, _i, _i, _vp, _vp], _i),
    "moe_repack_w4": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp], _i),
    "moe_expert_gemm_w4": ([_i, _i, _vp, _i, _i, _i, _i, _i] + [_vp] * 5 + [_i, _vp, _vp], _i),
    "moe_combine": ([_vp, _vp, _vp, _vp, _i, _i, _i, _vp], _i),
    "moe_decode_workspace_size": ([_i, _i], _sz),
    "moe_layer_forward": ([_vp, _vp, _vp] + [_i] * 7 + [ctypes.POINTER(Weights), ctypes.POINTER(Buffers), _vp], _i),
    "moe_layer_forward_host": ([_vp] * 6 + [_i] * 7 + [ctypes.POINTER(Weights), ctypes.POINTER(Buffers), _vp], _i),
    "moe_get_device_error": ([ctypes.POINTER(ctypes.c_int32)], _i),
    "moe_set_wait_limit_ns": ([ctypes.c_uint64], None),
    "moe_trace_words": ([], ctypes.c_size_t),
    "moe_trace_reset": ([_vp], _i),
    "moe_trace_read": ([_vp, ctypes.c_size_t], _i),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise OSError(f"{path} is missing: build it with `python -m bit_mixture_experts_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != MOE_OK:
        raise MoeError(name, rc)
    return rc


def _ptr(t):
    """A tensor's data pointer, or a raw address given as an int (every entry point declares its
    pointer arguments as void*, so ctypes takes the integer as it is)."""
    if t is None or isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


# --------------------------------------------------------------------------- #
# thin wrappers with the C names
# --------------------------------------------------------------------------- #
def moe_version() -> int:
    return load().moe_version()


def moe_launch_count() -> int:
    return load().moe_launch_count()


def moe_block_map_capacity(T, E, k, block_n) -> int:
    return load().moe_block_map_capacity(T, E, k, block_n)


def moe_route_workspace_size(T, E, k, block_n) -> int:
    return load().moe_route_workspace_size(T, E, k, block_n)


def moe_repacked_bytes(n_mat, rows, K) -> int:
    return load().moe_repacked_bytes(n_mat, rows, K)


def moe_route(logits, k, block_n, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks,
              workspace, stream=None):
    T, E = logits.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("moe_route", _ptr(logits), T, E, k, block_n, _ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets),
          _ptr(perm), _ptr(inv_perm), _ptr(block_map), _ptr(num_blocks), _ptr(workspace), ws_bytes, _stream(stream))


def moe_route_x(x, w_router, k, block_n, logits, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map,
                num_blocks, workspace, stream=None):
    """Router projection fused with the top-k (x bf16 [T, H], w_router bf16 [E, H] -> logits), then routing."""
    T, H = x.shape
    E = w_router.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("moe_route_x", _ptr(x), _ptr(w_router), T, H, E, k, block_n, _ptr(logits), _ptr(topk_ids), _ptr(topk_w),
          _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(block_map), _ptr(num_blocks),
          _ptr(workspace), ws_bytes, _stream(stream))


def moe_router(x, w_router, k, logits, topk_ids, topk_w, stream=None):
    """Router projection and top-k only (x bf16 [T, H], w_router bf16 [E, H] -> logits, ids, weights)."""
    T, H = x.shape
    E = w_router.shape[0]
    _call("moe_router", _ptr(x), _ptr(w_router), T, H, E, k, _ptr(logits), _ptr(topk_ids), _ptr(topk_w),
          _stream(stream))


def moe_rms_norm(x, out, eps=1e-6, stream=None):
    """out = bf16(x / rms(x)) per token (x, out bf16 [T, H] on the device)."""
    T, H = x.shape
    _call("moe_rms_norm", _ptr(x), _ptr(out), T, H, float(eps), _stream(stream))


def moe_norm_router(x, w_router, x_norm, logits, eps=1e-6, stream=None):
    """Decode step (T <= 8): x_norm = rms_norm(x) and logits = x_norm w_router^T in one launch."""
    T, H = x.shape
    E = w_router.shape[0]
    _call("moe_norm_router", _ptr(x), _ptr(w_router), T, H, E, float(eps), _ptr(x_norm), _ptr(logits),
          _stream(stream))


def moe_route_noalloc(logits, k, block_n, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks,
                      stream=None):
    """moe_route with the library's own fixed scratch instead of a workspace (no allocation)."""
    T, E = logits.shape
    _call("moe_route_noalloc", _ptr(logits), T, E, k, block_n, _ptr(topk_ids), _ptr(topk_w), _ptr(counts),
          _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(block_map), _ptr(num_blocks), _stream(stream))


def moe_repack_w4(packed, scale, bias, gate_up, out, stream=None):
    n_mat, rows, kw = packed.shape
    _call("moe_repack_w4", _ptr(packed), _ptr(scale), _ptr(bias), n_mat, rows, kw * 8, int(gate_up), _ptr(out),
          _stream(stream))


def moe_expanded_bytes(n_mat, rows, K) -> int:
    return load().moe_expanded_bytes(n_mat, rows, K)


def moe_expand_w4(w_repacked, n_mat, rows, K, out, stream=None):
    """The unfused path's bf16 copy of repacked 4-bit weights (for IMPL_TC_BF16)."""
    _call("moe_expand_w4", _ptr(w_repacked), n_mat, rows, K, _ptr(out), _stream(stream))


def moe_expert_gemm_w4(mode, impl, act, T, H, F, E, k, w_packed, perm, topk_w, block_map, num_blocks, block_n, out,
                       stream=None):
    _call("moe_expert_gemm_w4", mode, impl, _ptr(act), T, H, F, E, k, _ptr(w_packed), _ptr(perm), _ptr(topk_w),
          _ptr(block_map), _ptr(num_blocks), block_n, _ptr(out), _stream(stream))


def moe_combine(y, inv_perm, topk_w, out, stream=None):
    """out[t] = bf16(sum_j topk_w[t, j] * y[inv_perm[t*k + j]] + y[A + t]); y bf16 [A+T, H]."""
    T, k = topk_w.shape
    H = out.shape[1]
    _call("moe_combine", _ptr(y), _ptr(inv_perm), _ptr(topk_w), _ptr(out), T, H, k, _stream(stream))


def moe_expert_ffn_w4(x, T, H, F, E, k, w13, w2, perm, block_map, num_blocks, block_n, y, stream=None):
    """Both projections per expert tile in one launch, h kept on chip (y written, no h)."""
    _call("moe_expert_ffn_w4", _ptr(x), T, H, F, E, k, _ptr(w13), _ptr(w2), _ptr(perm), _ptr(block_map),
          _ptr(num_blocks), block_n, _ptr(y), _stream(stream))


def moe_down_combine_workspace_size(T, H) -> int:
    return int(load().moe_down_combine_workspace_size(T, H))


def moe_down_combine(h, T, H, F, E, k, w_packed, perm, inv_perm, topk_w, block_map, num_blocks, block_n, y, out,
                     workspace, stream=None):
    """The down GEMM with the combine in its epilogue (y and out written; workspace zero-filled once)."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _call("moe_down_combine", _ptr(h), T, H, F, E, k, _ptr(w_packed), _ptr(perm), _ptr(inv_perm), _ptr(topk_w),
          _ptr(block_map), _ptr(num_blocks), block_n, _ptr(y), _ptr(out), _ptr(workspace), ws_bytes,
          _stream(stream))


def moe_decode_workspace_size(T, H) -> int:
    return int(load().moe_decode_workspace_size(T, H))


def moe_layer_forward(x, logits, out, T, H, F, E, k, block_n, impl, weights: Weights, buffers: Buffers,
                      stream=None):
    _call("moe_layer_forward", _ptr(x), _ptr(logits), _ptr(out), T, H, F, E, k, block_n, impl,
          ctypes.byref(weights), ctypes.byref(buffers), _stream(stream))


def moe_layer_forward_host(x_host, logits_host, out_host, x_dev, logits_dev, out_dev, T, H, F, E, k, block_n, impl,
                           weights: Weights, buffers: Buffers, stream=None):
    _call("moe_layer_forward_host", _ptr(x_host), _ptr(logits_host), _ptr(out_host), _ptr(x_dev), _ptr(logits_dev),
          _ptr(out_dev), T, H, F, E, k, block_n, impl, ctypes.byref(weights), ctypes.byref(buffers),
          _stream(stream))


def moe_set_wait_limit_ns(ns: int) -> None:
    load().moe_set_wait_limit_ns(int(ns))


def moe_trace_words() -> int:
    """Words of wait statistics the loaded library keeps (0 unless it is the trace build)."""
    return int(load().moe_trace_words())


def moe_trace_reset(stream=None) -> None:
    _call("moe_trace_reset", _stream(stream))


def moe_trace_read(out) -> None:
    """Copies the wait statistics into `out`, a contiguous uint64 numpy array of moe_trace_words() words."""
    _call("moe_trace_read", out.ctypes.data, out.size)


def moe_get_device_error() -> int:
    code = ctypes.c_int32(0)
    _call("moe_get_device_error", ctypes.byref(code))
    return code.value
