"""moe_route_noalloc, the routing entry point for callers that may not allocate
device memory (a host engine that owns the whole device, or a latency path
that cannot afford cudaMalloc's implicit synchronisation): its outputs must
equal moe_route's, which uses a caller-provided workspace, and the oracle's,
on two calls in a row.  The second call is smaller than the first, so it runs
over the counts the first call left in the library's fixed scratch array.  A
call after calls whose grid barrier gave up (a wait limit far too short) must
be correct again, and so must the single-CTA path that uses no scratch.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here."""
import numpy as np
import pytest

import workloads

import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _buffers(T, E, k, bn, dev):
    import torch
    from bit_mixture_experts_gb300 import _lib
    A = T * k
    cap = _lib.moe_block_map_capacity(T, E, k, bn)
    return {
        "topk_ids": torch.full((T, k), -7, dtype=torch.int32, device=dev),
        "topk_w": torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
        "inv_perm": torch.full((A,), -7, dtype=torch.int32, device=dev),
        "block_map": torch.full((cap, 3), -7, dtype=torch.int32, device=dev),
        "num_blocks": torch.full((1,), -7, dtype=torch.int32, device=dev),
    }


def _route_both(logits_np, k, bn):
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    T, E = logits_np.shape
    logits = torch.from_numpy(np.ascontiguousarray(logits_np, np.float32)).to(dev)
    ref = _buffers(T, E, k, bn, dev)
    got = _buffers(T, E, k, bn, dev)
    # moe_route needs its workspace zero-filled before the first call (its barrier counters start at zero)
    ws = torch.zeros(max(_lib.moe_route_workspace_size(T, E, k, bn), 16), dtype=torch.uint8, device=dev)
    _lib.moe_route(logits, k, bn, *(ref[n] for n in ("topk_ids", "topk_w", "counts", "offsets", "perm",
                                                     "inv_perm", "block_map", "num_blocks")), ws)
    _lib.moe_route_noalloc(logits, k, bn, *(got[n] for n in ("topk_ids", "topk_w", "counts", "offsets", "perm",
                                                             "inv_perm", "block_map", "num_blocks")))
    torch.cuda.synchronize()
    assert _lib.moe_get_device_error() == 0
    return ({n: v.cpu().numpy() for n, v in ref.items()}, {n: v.cpu().numpy() for n, v in got.items()})


def _assert_oracle(logits_np, k, bn, got):
    from oracle import moe_ref
    ref = moe_ref.route(logits_np, k, bn)
    for n in ("topk_ids", "counts", "offsets", "perm", "inv_perm"):
        assert np.array_equal(got[n], ref[n]), n
    nb = int(got["num_blocks"][0])
    assert nb == ref["num_blocks"]
    assert np.array_equal(got["block_map"][:nb], ref["block_map"])
    assert np.allclose(got["topk_w"], ref["topk_w"], rtol=1e-6, atol=float(np.finfo(np.float32).tiny))


def _assert_same(ref, got):
    nb = int(ref["num_blocks"][0])
    assert int(got["num_blocks"][0]) == nb
    for n in ("topk_ids", "counts", "offsets", "perm", "inv_perm"):
        assert np.array_equal(got[n], ref[n]), n
    assert np.array_equal(got["block_map"][:nb], ref["block_map"][:nb])
    assert np.allclose(got["topk_w"], ref["topk_w"], rtol=1e-6, atol=float(np.finfo(np.float32).tiny))


def test_noalloc_matches_workspace_route_twice():
    """Two calls in a row (4096 then 512 tokens, both over 256 experts) equal moe_route's outputs."""
    shape = workloads.FULL
    for T in (4096, 512):
        tok = workloads.make_tokens(shape, T, seed=5)
        ref, got = _route_both(tok["logits"], shape.k, 256)
        _assert_same(ref, got)
        _assert_oracle(tok["logits"], shape.k, 256, got)


def test_noalloc_single_cta_path():
    """64 tokens x top-8 (512 assignments): the one-CTA routing kernel, which needs no scratch."""
    shape = workloads.FULL
    tok = workloads.make_tokens(shape, 64, seed=6)
    ref, got = _route_both(tok["logits"], shape.k, 64)
    _assert_same(ref, got)
    _assert_oracle(tok["logits"], shape.k, 64, got)


def test_noalloc_correct_after_barrier_gave_up():
    """Calls whose grid barrier ran out of time (0.2 us limit) leave nothing behind that breaks the
    next call: its barrier counters are cleared before it starts."""
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    shape = workloads.FULL
    T, k, bn = 4096, shape.k, 128
    tok = workloads.make_tokens(shape, T, seed=7)
    logits = torch.from_numpy(tok["logits"]).to(dev)
    b = _buffers(T, shape.E, k, bn, dev)
    names = ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv_perm", "block_map", "num_blocks")
    _lib.moe_set_wait_limit_ns(200)
    try:
        for _ in range(5):
            _lib.moe_route_noalloc(logits, k, bn, *(b[n] for n in names))
            torch.cuda.synchronize()
            _lib.moe_get_device_error()  # a timeout or an inconsistent count may be reported; cleared here
    finally:
        _lib.moe_set_wait_limit_ns(1_000_000_000)
    ref, got = _route_both(tok["logits"], k, bn)
    _assert_same(ref, got)
    _assert_oracle(tok["logits"], k, bn, got)


def test_noalloc_rejects_more_experts_than_its_scratch():
    import torch
    from bit_mixture_experts_gb300 import _lib
    dev = G.torch_dev()
    T, E, k, bn = 4096, 512, 8, 128         # 256 chunks x 512 experts of counts: 512 KiB, beyond the 256 KiB
    assert _lib.moe_route_workspace_size(T, E, k, bn) > 256 * 1024
    logits = torch.zeros((T, E), dtype=torch.float32, device=dev)
    b = _buffers(T, E, k, bn, dev)
    with pytest.raises(_lib.MoeError) as ex:
        _lib.moe_route_noalloc(logits, k, bn, *(b[n] for n in ("topk_ids", "topk_w", "counts", "offsets", "perm",
                                                               "inv_perm", "block_map", "num_blocks")))
    assert ex.value.code == -4
