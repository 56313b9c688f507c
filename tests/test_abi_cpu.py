"""The C-ABI library on the CPU: it loads, exports every entry point that
include/moe_w4.h declares, and its host-only paths (sizes, argument checks
that fail before any CUDA call) behave as documented.  No compute runs."""
import ctypes
import os
import re

import pytest

from oracle import moe_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_mixture_experts_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    from bit_mixture_experts_gb300 import _lib
    decl = declared_symbols()
    assert len(decl) >= 11
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(_lib.SYMBOLS)


def test_version(lib):
    assert lib.moe_version() == 0x000100


@pytest.mark.parametrize("T,E,k,bn", [(1, 16, 2, 128), (512, 256, 8, 128), (4096, 256, 8, 256), (7, 3, 3, 2)])
def test_block_map_capacity_matches_oracle(lib, T, E, k, bn):
    assert lib.moe_block_map_capacity(T, E, k, bn) == moe_ref.block_map_capacity(T, E, k, bn)


def test_workspace_size(lib):
    assert lib.moe_route_workspace_size(1, 256, 8, 128) == 0          # single-CTA path needs none
    assert lib.moe_route_workspace_size(4096, 256, 8, 128) > 0
    assert lib.moe_route_workspace_size(4096, 256, 8, 128) % 16 == 0


def _route(lib, T=8, E=16, k=2, bn=128, ptr=16, ws=0):
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    return lib.moe_route(p, T, E, k, bn, p, p, p, p, p, p, p, p, p, ws, None)


def test_route_argument_errors(lib):
    assert _route(lib, T=0) == -3
    assert _route(lib, k=17, E=16) == -3
    assert _route(lib, k=33, E=64) == -3
    assert _route(lib, E=1025) == -3
    assert _route(lib, bn=0) == -3
    assert _route(lib, ptr=None) == -1
    assert _route(lib, ptr=8) == -2
    assert _route(lib, T=4096, E=256, k=8, ptr=16, ws=0) == -4


def test_gemm_argument_errors(lib):
    p = ctypes.c_void_p(256)
    args = lambda mode, impl, H, F, bn, ptr=p: lib.moe_expert_gemm_w4(
        mode, impl, ptr, 16, H, F, 8, 2, ptr, ptr, ptr, ptr, ptr, bn, ptr, None)
    assert args(0, 2, 100, 128, 128) == -3      # H % 64
    assert args(0, 2, 128, 96, 128) == -3       # F % 64
    assert args(0, 2, 192, 128, 128) == -3      # H % 128 (tensor-core kernel)
    assert args(1, 3, 128, 192, 8) == -3        # F % 128 (GEMV kernel)
    assert args(0, 2, 128, 128, 129) == -3      # tile height above the tensor-core kernel's 128
    assert args(0, 3, 128, 128, 9) == -3        # tile height above the GEMV kernel's 8
    assert args(5, 2, 128, 128, 128) == -7      # mode
    assert args(0, 1, 128, 128, 128) == -7      # no kernel 1 (the CUDA-core GEMM is not part of the library)
    assert args(0, 2, 128, 128, 128, ptr=None) == -1
    assert args(0, 2, 128, 128, 128, ptr=ctypes.c_void_p(260)) == -2


def test_combine_argument_errors(lib):
    p = ctypes.c_void_p(16)
    assert lib.moe_combine(p, p, p, p, 4, 100, 2, None) == -3       # H % 8
    assert lib.moe_combine(p, p, p, p, 4, 128, 0, None) == -3       # k < 1
    assert lib.moe_combine(p, p, p, p, 4, 128, 33, None) == -3      # k > 32
    assert lib.moe_combine(None, p, p, p, 4, 128, 2, None) == -1
    assert lib.moe_combine(p, p, ctypes.c_void_p(20), p, 4, 128, 2, None) == -2


def test_down_combine_argument_errors(lib):
    p = ctypes.c_void_p(256)
    ws = lib.moe_down_combine_workspace_size(16, 256)
    assert ws == 16 * 2 * 4
    assert lib.moe_down_combine_workspace_size(16, 192) == 0
    assert lib.moe_down_combine_workspace_size(0, 256) == 0
    args = lambda H, F, bn, ptr=p, wsb=ws: lib.moe_down_combine(
        ptr, 16, H, F, 8, 2, ptr, ptr, ptr, ptr, ptr, ptr, bn, ptr, ptr, ptr, wsb, None)
    assert args(192, 128, 128) == -3            # H % 128
    assert args(256, 192, 128) == -3            # F % 128
    assert args(256, 128, 129) == -3            # tile height above 128
    assert args(256, 128, 128, ptr=None) == -1
    assert args(256, 128, 128, ptr=ctypes.c_void_p(260)) == -2
    assert args(256, 128, 128, wsb=ws - 4) == -4


def test_expert_ffn_argument_errors(lib):
    p = ctypes.c_void_p(256)
    args = lambda H, F, bn, ptr=p: lib.moe_expert_ffn_w4(ptr, 16, H, F, 8, 2, ptr, ptr, ptr, ptr, ptr, bn, ptr, None)
    assert args(192, 256, 64) == -3             # H % 128
    assert args(256, 384, 64) == -3             # F % 256
    assert args(256, 256, 65) == -3             # tiles above 64 rows (h must fit in shared memory)
    assert args(256, 256, 64, ptr=None) == -1
    assert args(256, 256, 64, ptr=ctypes.c_void_p(260)) == -2


def test_repacked_bytes(lib):
    # one 4608-byte block (2 halves x 128 rows x 16 B of nibbles, then 128 x (scale, bias)) per
    # 128-row tile and 64-wide K group: exactly the bytes of the canonical layout of the matrix
    assert lib.moe_repacked_bytes(1, 128, 64) == 4608
    assert lib.moe_repacked_bytes(1, 1024, 2048) == 1_179_648     # gate/up of one expert, H=2048 F=512
    assert lib.moe_repacked_bytes(1, 2048, 512) == 589_824        # down of one expert
    for n, rows, K in ((3, 1024, 2048), (17, 256, 256), (2, 2048, 512)):
        canonical = rows * (K // 8) * 4 + 2 * rows * (K // 64) * 2   # packed words + bf16 scale and bias
        assert lib.moe_repacked_bytes(n, rows, K) == n * canonical
    assert lib.moe_repacked_bytes(1, 100, 2048) == 0
    assert lib.moe_repacked_bytes(1, 128, 96) == 0
    assert lib.moe_repacked_bytes(0, 128, 64) == 0


def test_decode_workspace_size(lib):
    for T in range(1, 9):
        n = lib.moe_decode_workspace_size(T, 2048)
        assert n > 0 and n % 4 == 0
    assert lib.moe_decode_workspace_size(0, 2048) == 0
    assert lib.moe_decode_workspace_size(9, 2048) == 0          # above the fused path's 8 tokens


def test_repack_argument_errors(lib):
    p = ctypes.c_void_p(256)
    rp = lambda rows, K, gate_up, ptr=p: lib.moe_repack_w4(ptr, ptr, ptr, 2, rows, K, gate_up, ptr, None)
    assert rp(100, 2048, 0) == -3
    assert rp(128, 96, 0) == -3
    assert rp(128, 2048, 1) == -3       # gate/up tile pairs need rows / 2 % 128 == 0
    assert rp(256, 2048, 1, ptr=None) == -1
    assert rp(256, 2048, 1, ptr=ctypes.c_void_p(264)) == -2


def test_route_noalloc_argument_errors(lib):
    p = ctypes.c_void_p(16)
    r = lambda T=8, E=16, k=2, bn=128, ptr=p: lib.moe_route_noalloc(ptr, T, E, k, bn, *([ptr] * 8), None)
    assert r(T=0) == -3
    assert r(k=17, E=16) == -3
    assert r(bn=0) == -3
    assert r(ptr=None) == -1
    assert r(ptr=ctypes.c_void_p(8)) == -2
    # per-chunk counts of 256 chunks x 1024 experts exceed the library's fixed 256 KiB array
    assert lib.moe_route_workspace_size(1 << 20, 1024, 8, 128) > 256 * 1024
    assert r(T=1 << 20, E=1024, k=8) == -4


def test_layer_forward_argument_errors(lib):
    from bit_mixture_experts_gb300 import _lib
    p = 256
    w = _lib.Weights(p, p)
    small_ws = _lib.Buffers(*([p] * 10), p, 0, p, 1)            # decode workspace of 1 byte
    fwd = lambda T, H, bufs, weights=w: lib.moe_layer_forward(
        ctypes.c_void_p(p), ctypes.c_void_p(p), ctypes.c_void_p(p), T, H, 512, 256, 8, 8, 3,
        ctypes.byref(weights) if weights is not None else None, ctypes.byref(bufs) if bufs is not None else None,
        None)
    assert fwd(1, 2048, None) == -1
    assert fwd(1, 2048, small_ws, weights=None) == -1
    assert fwd(1, 100, small_ws) == -3                          # H % 64 on the fused decode path
    assert fwd(1, 2048, small_ws) == -4                         # decode workspace below its size


def test_product_library_records_no_trace(lib):
    """Wait statistics exist only in the trace build; the product library says so and records nothing."""
    import numpy as np
    assert lib.moe_trace_words() == 0
    assert lib.moe_trace_reset(None) == -7
    buf = np.zeros(4, np.uint64)
    assert lib.moe_trace_read(buf.ctypes.data, buf.size) == -7


def test_trace_build_exports_its_words():
    """The -DMOE_TRACE build of the same sources (libmoe_w4_trace.so) compiles, loads beside the product
    library, and keeps 1024 CTAs x 32 warps x 4 words."""
    from bit_mixture_experts_gb300 import build
    path = build.build(trace=True)
    assert os.path.basename(path) == "libmoe_w4_trace.so"
    tl = ctypes.CDLL(path)
    tl.moe_trace_words.restype = ctypes.c_size_t
    assert tl.moe_trace_words() == 1024 * 32 * 4
    tl.moe_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    assert tl.moe_trace_read(None, 4) == -1  # MOE_ERR_NULL before any CUDA call
