"""GPU routing (moe_route through the C ABI) against the oracle: bit-exact ids,
counts, offsets, permutation, inverse permutation, block map and tile count;
renormalised weights within 1e-6 relative."""
import numpy as np
import pytest

import workloads
from oracle import moe_ref

import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_route(logits_np, k, bn):
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    T, E = logits_np.shape
    A = T * k
    logits = torch.from_numpy(np.ascontiguousarray(logits_np, np.float32)).to(dev)
    cap = _lib.moe_block_map_capacity(T, E, k, bn)
    wsb = _lib.moe_route_workspace_size(T, E, k, bn)
    o = {
        "topk_ids": torch.full((T, k), -7, dtype=torch.int32, device=dev),
        "topk_w": torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
        "inv_perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
        "block_map": torch.full((cap, 3), -7, dtype=torch.int32, device=dev),
        "num_blocks": torch.full((1,), -7, dtype=torch.int32, device=dev),
    }
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
    _lib.moe_route(logits, k, bn, o["topk_ids"], o["topk_w"], o["counts"], o["offsets"], o["perm"],
                   o["inv_perm"], o["block_map"], o["num_blocks"], ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    return {n: v.cpu().numpy() for n, v in o.items()}


def check_route(logits, k, bn):
    ref = moe_ref.route(logits, k, bn)
    got = run_route(logits, k, bn)
    assert np.array_equal(got["topk_ids"], ref["topk_ids"])
    # 1e-6 relative; weights below float32's normal range (exp(-87) and less) are
    # compared absolutely, since a subnormal float32 cannot hold 1e-6 relative
    assert np.allclose(got["topk_w"], ref["topk_w"], rtol=1e-6, atol=float(np.finfo(np.float32).tiny))
    assert np.array_equal(got["counts"], ref["counts"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["perm"], ref["perm"])
    assert np.array_equal(got["inv_perm"], ref["inv_perm"])
    nb = int(got["num_blocks"][0])
    assert nb == ref["num_blocks"]
    assert np.array_equal(got["block_map"][:nb], ref["block_map"])
    return got


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode8", "prefill512", "prefill4k", "skew16k"])
@pytest.mark.parametrize("bn", [128, 256])
def test_route_workloads(name, bn):
    wl = workloads.WORKLOADS[name]
    tok = workloads.make_tokens(wl.shape, wl.T, 0, wl.skew)
    check_route(tok["logits"], wl.shape.k, bn)


@pytest.mark.parametrize("T,E,k,bn", [(1, 16, 2, 16), (37, 16, 2, 8), (300, 64, 8, 32), (129, 256, 8, 256),
                                      (1000, 32, 1, 64), (200, 512, 16, 48), (64, 1024, 32, 128),
                                      (2049, 8, 8, 128), (5000, 256, 8, 1), (20, 1024, 16, 64)])
def test_route_shapes(T, E, k, bn):
    r = np.random.default_rng(T + E)
    check_route(r.standard_normal((T, E)).astype(np.float32), k, bn)


def test_route_ties_and_signed_zero():
    """Equal logits (including -0.0 against +0.0) go to the lower expert index."""
    r = np.random.default_rng(9)
    lg = np.round(r.standard_normal((700, 64)) * 2).astype(np.float32)
    lg[::7] = 0.0
    lg[1::7] = -0.0
    lg[2::7, ::2] = -0.0
    got = check_route(lg, 8, 128)
    assert got["topk_ids"][0].tolist() == list(range(8))


def test_route_hot_expert():
    """Every token prefers expert 3: one expert with T rows and many tiles."""
    r = np.random.default_rng(10)
    lg = r.standard_normal((3000, 256)).astype(np.float32)
    lg[:, 3] += 100.0
    check_route(lg, 8, 128)


def test_route_deterministic():
    wl = workloads.WORKLOADS["prefill4k"]
    tok = workloads.make_tokens(wl.shape, wl.T, 0)
    a = run_route(tok["logits"], 8, 256)
    b = run_route(tok["logits"], 8, 256)
    for n in a:
        assert np.array_equal(a[n], b[n]), n


def test_route_reports_a_workspace_that_was_not_zeroed():
    """A workspace holding stale bytes (here 0x01 in every byte: the barrier counter already
    past the chunk count, per-chunk counts that cannot come from the call) makes moe_route
    report MOE_DEV_BAD_WORKSPACE.  Without the barrier the chunks' counts may or may not be
    complete when they are summed; a CTA that finds them inconsistent writes nothing from them,
    one that finds them complete writes the true result, so every output entry is either
    untouched or in range.  With a zero-filled workspace the outputs are exact again."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    wl = workloads.WORKLOADS["prefill512"]
    tok = workloads.make_tokens(wl.shape, wl.T, 0, wl.skew)
    T, E, k, bn = wl.T, wl.shape.E, wl.shape.k, 64
    logits = torch.from_numpy(np.ascontiguousarray(tok["logits"], np.float32)).to(dev)
    A = T * k
    cap = _lib.moe_block_map_capacity(T, E, k, bn)
    o = {"topk_ids": torch.full((T, k), -7, dtype=torch.int32, device=dev),
         "topk_w": torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
         "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
         "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
         "perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
         "inv_perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
         "block_map": torch.full((cap, 3), -7, dtype=torch.int32, device=dev),
         "num_blocks": torch.full((1,), -7, dtype=torch.int32, device=dev)}
    names = ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv_perm", "block_map", "num_blocks")
    wsb = max(_lib.moe_route_workspace_size(T, E, k, bn), 16)
    assert wsb > 16  # the multi-CTA path, which has the barrier
    _lib.moe_get_device_error()  # clear
    ws = torch.full((wsb,), 1, dtype=torch.uint8, device=dev)
    _lib.moe_route(logits, k, bn, *(o[n] for n in names), ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 4  # MOE_DEV_BAD_WORKSPACE
    perm = o["perm"].cpu().numpy()
    assert np.all((perm == -7) | ((perm >= 0) & (perm < A)))
    nb = int(o["num_blocks"].item())
    assert nb == -7 or 0 < nb <= cap
    ws.zero_()
    _lib.moe_route(logits, k, bn, *(o[n] for n in names), ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    ref = moe_ref.route(tok["logits"], k, bn)
    assert np.array_equal(o["perm"].cpu().numpy(), ref["perm"])
    assert int(o["num_blocks"].item()) == ref["num_blocks"]


def test_route_one_workspace_for_two_token_counts():
    """One zero-filled workspace sized for 4096 tokens serves a 4096-token call and then a
    512-token call: the counters sit in the workspace's last 16 bytes, away from the per-chunk
    counts the larger call left behind."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    shape = workloads.FULL
    E, k, bn = shape.E, shape.k, 128
    ws = torch.zeros(_lib.moe_route_workspace_size(4096, E, k, bn), dtype=torch.uint8, device=dev)
    names = ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv_perm", "block_map", "num_blocks")
    _lib.moe_get_device_error()
    for T in (4096, 512):
        tok = workloads.make_tokens(shape, T, seed=3)
        A = T * k
        cap = _lib.moe_block_map_capacity(T, E, k, bn)
        o = {"topk_ids": torch.full((T, k), -7, dtype=torch.int32, device=dev),
             "topk_w": torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
             "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
             "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
             "perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
             "inv_perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
             "block_map": torch.full((cap, 3), -7, dtype=torch.int32, device=dev),
             "num_blocks": torch.full((1,), -7, dtype=torch.int32, device=dev)}
        logits = torch.from_numpy(np.ascontiguousarray(tok["logits"], np.float32)).to(dev)
        _lib.moe_route(logits, k, bn, *(o[n] for n in names), ws)
        torch.cuda.synchronize()
        assert _lib.moe_get_device_error() == 0
        ref = moe_ref.route(tok["logits"], k, bn)
        assert np.array_equal(o["perm"].cpu().numpy(), ref["perm"])
        nb = int(o["num_blocks"].item())
        assert nb == ref["num_blocks"]
        assert np.array_equal(o["block_map"].cpu().numpy()[:nb], ref["block_map"])
