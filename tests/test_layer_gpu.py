"""The whole layer on the GPU (moe_layer_forward through the C ABI) against the
float64 oracle with the complete check of tests/parity.py (routing bit-exact,
every h and y a valid rounding, every output within 1e-2 + 1e-2|ref|): all
tokens on shapes the oracle finishes in seconds and on the 512-token prefill,
and one token per block-map tile (so every tile, ragged tails included, is
checked at full width) on the other full-size workloads."""
import numpy as np
import pytest

from oracle import moe_ref

import gpu_util as G

pytestmark = pytest.mark.gpu

IMPLS = ["tc", "tc2", "gemv"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_layer(d, impl, block_n=None, reps=1):
    """Layer forward(s) through the C ABI; returns the outputs (float64) and the layer."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    wl = d["workload"]
    s = wl.shape
    layer = MoELayerW4(s.H, s.E, s.k, s.F, d, impl=impl, block_n=block_n)
    x, logits = G.to_dev_inputs(d)
    outs = []
    for _ in range(reps):
        outs.append(layer.forward(x, logits).clone())
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    return [G.bf16_to_f64(o) for o in outs], layer


SMALL = [
    (64, 256, 16, 2, 128, False),     # the tiny workload's shape
    (300, 512, 32, 4, 256, False),    # ragged tiles, several shared-expert tiles
    (512, 256, 8, 2, 128, False),     # experts above one tile
    (1, 256, 16, 2, 128, False),      # a single token
    (77, 128, 64, 8, 128, False),     # many empty experts
    (1000, 256, 16, 4, 384, True),    # skewed logits (Zipf offset), F not a power of two
    (600, 256, 8, 2, 256, False),     # 128-row tiles, F % 256 == 0: down units of one M-tile, 4-group stages
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("spec", SMALL, ids=lambda s: "T{}_H{}_E{}_k{}_F{}{}".format(*s[:5], "_skew" if s[5] else ""))
def test_layer_small(spec, impl):
    d = G.workload(spec)
    (got,), layer = run_layer(d, impl)
    G.check_layer(d, layer, got, what=f"layer {spec} {impl}")


@pytest.mark.parametrize("block_n", [16, 48, 64, 96, 128])
def test_layer_tc_block_sizes(block_n):
    """The tensor-core kernel with every tile height it supports (N = rows rounded up to 16)."""
    spec = (700, 256, 16, 4, 128, False)
    d = G.workload(spec)
    (got,), layer = run_layer(d, "tc", block_n=block_n)
    G.check_layer(d, layer, got, what=f"tc block_n={block_n}")


@pytest.mark.parametrize("impl", IMPLS)
def test_layer_repeatable(impl):
    """Two calls in a row give the same result (the accumulator is left zero)."""
    d = G.workload((300, 512, 32, 4, 256, False))
    (a, b), layer = run_layer(d, impl, reps=2)
    G.check_layer(d, layer, a, what="first call")
    G.check_layer(d, layer, b, what="second call")


@pytest.mark.parametrize("block_n", [32, 64, 96, 128, 160, 192, 224, 256])
def test_layer_tc2_block_sizes(block_n):
    """The CTA-pair kernel with tile heights across its range (N = rows rounded up to 32, half in each
    CTA): four-group stages up to 128 rows, two accumulator buffers up to 192, one above."""
    spec = (700, 256, 16, 4, 128, False)
    d = G.workload(spec)
    (got,), layer = run_layer(d, "tc2", block_n=block_n)
    G.check_layer(d, layer, got, what=f"tc2 block_n={block_n}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["decode1", "decode8", "prefill512", "prefill4k", "skew16k"])
def test_layer_full_size_every_tile(name, impl):
    """Full-size workloads: every output of one token per block-map tile (the token of each tile's
    last row, read from the GPU's own block map), so every tile of every expert is checked."""
    import parity
    d = G.workload(name)
    wl = d["workload"]
    (got,), layer = run_layer(d, impl)
    a = G.gpu_arrays(layer, wl.T, got)
    toks = parity.tile_tokens(a["block_map"], a["num_blocks"], a["perm"], wl.T, wl.shape.k)
    G.check_layer(d, layer, got, tokens=toks, what=f"{name} {impl}, {toks.size} tokens (one per tile)")


@pytest.mark.parametrize("name", ["prefill4k", "skew16k"])
@pytest.mark.parametrize("block_n", [192, 256])
def test_layer_tc2_full_size_tall_tiles(name, block_n):
    """The CTA-pair kernel with 192- and 256-row tiles at full size, one token per tile."""
    import parity
    d = G.workload(name)
    wl = d["workload"]
    (got,), layer = run_layer(d, "tc2", block_n=block_n)
    a = G.gpu_arrays(layer, wl.T, got)
    toks = parity.tile_tokens(a["block_map"], a["num_blocks"], a["perm"], wl.T, wl.shape.k)
    G.check_layer(d, layer, got, tokens=toks, what=f"{name} tc2 block_n={block_n}, {toks.size} tokens (one per tile)")


@pytest.mark.parametrize("impl", IMPLS)
def test_layer_prefill512_all_outputs(impl):
    """The 512-token prefill through the full-width layer: every output element."""
    d = G.workload("prefill512")
    (got,), layer = run_layer(d, impl)
    G.check_layer(d, layer, got, what=f"prefill512 {impl}, all tokens")


@pytest.mark.parametrize("name", [(300, 512, 32, 4, 256, False), (600, 256, 8, 2, 256, False), "prefill512"],
                         ids=["T300", "T600", "prefill512"])
def test_unfused_path_equals_fused(name):
    """The unfused comparison path (weights expanded to a bf16 copy by moe_expand_w4, then the tensor-core
    kernel reading that copy) gives bit for bit the outputs of the fused kernel, and passes the oracle check."""
    d = G.workload(name)
    (fused,), _ = run_layer(d, "tc")
    (unfused,), layer = run_layer(d, "tc_bf16")
    assert np.array_equal(fused, unfused)
    G.check_layer(d, layer, unfused, what=f"unfused {name}")


@pytest.mark.parametrize("name", ["prefill4k"])
def test_unfused_path_full_size(name):
    """The unfused comparison path at 4096 tokens (128-row tiles, many work units per CTA, a weight ring
    of 32 KB stages): bit for bit the fused kernel's outputs, one token per tile against the oracle."""
    import parity
    d = G.workload(name)
    wl = d["workload"]
    (fused,), _ = run_layer(d, "tc")
    (unfused,), layer = run_layer(d, "tc_bf16")
    assert np.array_equal(fused, unfused)
    a = G.gpu_arrays(layer, wl.T, unfused)
    toks = parity.tile_tokens(a["block_map"], a["num_blocks"], a["perm"], wl.T, wl.shape.k)
    G.check_layer(d, layer, unfused, tokens=toks, what=f"unfused {name}, {toks.size} tokens (one per tile)")


@pytest.mark.parametrize("impl", IMPLS)
def test_gate_up_intermediate(impl):
    """The gate/up GEMM alone: h = bf16(silu(g) u) per permuted row against the oracle's h."""
    import torch

    import parity
    from bit_mixture_experts_gb300 import _lib
    from bit_mixture_experts_gb300.layer import MoELayerW4
    spec = (200, 256, 8, 2, 128, False)
    d = G.workload(spec)
    T, H, E, k, F = spec[:5]
    layer = MoELayerW4(H, E, k, F, d, impl=impl)
    x, logits = G.to_dev_inputs(d)
    b = layer.buffers(T)
    w = layer.weights
    bn = layer.block_n_for(T)
    _lib.moe_route(logits, k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                   b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
    b["h"].zero_()
    _lib.moe_expert_gemm_w4(_lib.GATE_UP, layer.impl_for(T), x, T, H, F, E, k, w.w13, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bn, b["h"])
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    got = G.bf16_to_f64(b["h"])
    perm = b["perm"].cpu().numpy()
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, k, want_h=True)
    ids = ref["topk_ids"].ravel()
    A = T * k
    want = np.zeros((A + T, F))
    for r in range(A):
        a = int(perm[r])
        want[r] = ref["h"][(a // k, int(ids[a]))]
    exact = np.zeros((A + T, F))
    for r in range(A):
        a = int(perm[r])
        exact[r] = ref["h_exact"][(a // k, int(ids[a]))]
    for t in range(T):
        want[A + t] = ref["h"][(t, E)]
        exact[A + t] = ref["h_exact"][(t, E)]
    # every h a valid rounding of its exact value (tests/parity.py): within the FP32 accumulation bound
    xs = moe_ref.bf16_value(d["x_bits"])
    delta = np.zeros_like(exact)
    w13s = {}
    for r in range(A + T):
        t, e = (r - A, E) if r >= A else (int(perm[r]) // k, int(ids[int(perm[r])]))
        if e not in w13s:
            w13s[e] = moe_ref.expert_weights(d, e)[0]
        w13 = w13s[e]
        g, u = xs[t] @ w13[:F].T, xs[t] @ w13[F:].T
        silu_g, slope = parity.silu_and_slope(g)
        delta[r] = (np.abs(slope * u) * parity.accumulation_bound(H, np.abs(xs[t]) @ np.abs(w13[:F]).T) +
                    np.abs(silu_g) * parity.accumulation_bound(H, np.abs(xs[t]) @ np.abs(w13[F:]).T) +
                    parity.EPI_REL * np.abs(exact[r]))
    ok, flip = parity.valid_rounding(got, exact, delta)
    assert ok.all(), f"h {impl}: {int((~ok).sum())} values are not a rounding of their exact value"
    assert np.array_equal(got[~flip], want[~flip])
    print(f"gate/up alone {impl}: {int(flip.sum())} of {flip.size} h round away from nearest (validated)")


DECODE = [
    (1, 256, 16, 2, 128, False),
    (5, 256, 16, 4, 128, False),
    (8, 128, 64, 8, 128, False),     # 64 assignments over 64 experts
    (8, 256, 16, 2, 256, True),      # skewed logits, F = 256
    (3, 128, 8, 8, 128, False),      # k = E: every expert in every token
    (8, 128, 32, 32, 128, False),    # k = 32: the largest assignment count of the fused path (256)
]


@pytest.mark.parametrize("spec", DECODE, ids=lambda s: "T{}_H{}_E{}_k{}_F{}{}".format(*s[:5], "_skew" if s[5] else ""))
def test_decode_fused(spec):
    """The fused decode kernel (T <= 8 with the GEMV kernel): every output against the oracle,
    and the routing it writes equal to moe_route's (bit-exact ids, counts, offsets,
    permutations, block map)."""
    d = G.workload(spec)
    T, H, E, k, F, _ = spec
    (got,), layer = run_layer(d, "gemv")
    G.check_layer(d, layer, got, what=f"fused decode {spec}")
    b = layer.buffers(T)
    assert b["decode_ws"] is not None
    ref = moe_ref.route(d["logits"], k, layer.block_n_for(T))
    assert np.array_equal(b["topk_ids"].cpu().numpy(), ref["topk_ids"])
    assert np.allclose(b["topk_w"].cpu().numpy(), ref["topk_w"], rtol=1e-6, atol=float(np.finfo(np.float32).tiny))
    for n in ("counts", "offsets", "perm", "inv_perm"):
        assert np.array_equal(b[n].cpu().numpy(), ref[n]), n
    nb = int(b["num_blocks"].item())
    assert nb == ref["num_blocks"]
    assert np.array_equal(b["block_map"].cpu().numpy()[:nb], ref["block_map"])


def test_decode_fused_repeatable():
    """Repeated fused calls (the kernel returns its counters to zero) give bit-identical outputs,
    equal to those of the four separate kernels."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    d = G.workload((8, 256, 16, 4, 128, False))
    outs, layer = run_layer(d, "gemv", reps=3)
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    assert int(layer.buffers(8)["decode_ws"].count_nonzero().item()) == 0
    # the unfused path: route, gate/up, down and combine launched one by one
    x, logits = G.to_dev_inputs(d)
    T, H, E, k, F = 8, 256, 16, 4, 128
    b = layer.buffers(T)
    w = layer.weights
    bn = layer.block_n_for(T)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _lib.moe_route(logits, k, bn, b["topk_ids"], b["topk_w"], b["counts"], b["offsets"], b["perm"],
                   b["inv_perm"], b["block_map"], b["num_blocks"], b["workspace"])
    _lib.moe_expert_gemm_w4(_lib.GATE_UP, _lib.IMPL_GEMV, x, T, H, F, E, k, w.w13, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bn, b["h"])
    _lib.moe_expert_gemm_w4(_lib.DOWN, _lib.IMPL_GEMV, b["h"], T, H, F, E, k, w.w2, b["perm"], b["topk_w"],
                            b["block_map"], b["num_blocks"], bn, b["y"])
    _lib.moe_combine(b["y"], b["inv_perm"], b["topk_w"], out)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    assert np.array_equal(G.bf16_to_f64(out), outs[0])
