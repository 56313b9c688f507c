"""The CPU oracle against its pins (brute force, closed forms, hand-derived goldens,
library routines, invariants), and mutation tests showing that a plausible
mistake planted in the oracle makes at least one pin fail."""
import numpy as np
import pytest

import workloads
from oracle import moe_ref

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_bruteforce_tiny_workload():
    """Vectorised oracle == per-token brute force on the 64-token tiny layer."""
    P.pin_bruteforce_layer()


def test_bruteforce_ragged_shape():
    P.pin_bruteforce_layer(shape=(128, 5, 3, 64), T=13, seed=3)


def test_bf16_floor_ceil():
    r = np.random.default_rng(11)
    a = r.standard_normal(5000) * 10.0 ** r.integers(-3, 3, 5000)
    lo, hi = moe_ref.bf16_floor_ceil(a)
    rn = moe_ref.round_bf16(a)
    assert np.all(lo <= a) and np.all(a <= hi)
    assert np.all((rn == lo) | (rn == hi))
    assert np.array_equal(moe_ref.round_bf16(lo), lo) and np.array_equal(moe_ref.round_bf16(hi), hi)
    # adjacent: nothing representable strictly between
    mid = 0.5 * (lo + hi)
    assert np.all((lo == hi) | ((moe_ref.round_bf16(mid) == lo) | (moe_ref.round_bf16(mid) == hi)))
    b = moe_ref.round_bf16(a)
    lo2, hi2 = moe_ref.bf16_floor_ceil(b)
    assert np.array_equal(lo2, b) and np.array_equal(hi2, b)


def test_intermediates_are_roundings_of_their_exact_values():
    """The h and y rows the oracle returns are the bf16 roundings of their exact values, and the
    layer output is the bf16 rounding of the weighted sum of its y rows."""
    d = workloads.make_workload(workloads.custom(9, 128, 4, 2, 64), 2)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, 2, want_h=True, want_y=True)
    for key, h in ref["h"].items():
        assert np.array_equal(h, moe_ref.round_bf16(ref["h_exact"][key]))
    for key, y in ref["y"].items():
        assert np.array_equal(y, moe_ref.round_bf16(ref["y_exact"][key]))
    acc = np.zeros_like(ref["out"])
    for t in range(9):
        for j in range(2):
            acc[t] += ref["topk_w"][t, j] * ref["y"][(t, int(ref["topk_ids"][t, j]))]
        acc[t] += ref["y"][(t, 4)]
    assert np.array_equal(ref["out"], moe_ref.round_bf16(acc))


def test_y_rounding_pinned_by_closed_form(monkeypatch):
    """Dropping the bf16 rounding of the down projection's output fails the scaled-down closed
    form (not only the brute force)."""
    monkeypatch.setattr(moe_ref, "down_output", lambda y: np.asarray(y, dtype=np.float64))
    with pytest.raises(AssertionError):
        P.pin_closed_form_scaled_down()


def test_skew_calibration():
    """The skewed long prefill leaves about 30 experts empty and one expert chosen by
    nearly every token (at most T of the T*k assignments can go to one expert)."""
    wl = workloads.WORKLOADS["skew16k"]
    tok = workloads.make_tokens(wl.shape, wl.T, 0, skew=True)
    ids, _ = moe_ref.topk_route(tok["logits"], wl.shape.k)
    counts = moe_ref.histogram(ids, wl.shape.E)
    assert 25 <= int((counts == 0).sum()) <= 35
    assert counts.max() > 0.9 * wl.T


def test_generator_statistics():
    wl = workloads.WORKLOADS["tiny"]
    d = workloads.make_workload(wl)
    x = workloads.bf16_bits_to_f32(d["x_bits"])
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1) < 0.05
    assert abs(d["logits"].std() - 1) < 0.1
    q = moe_ref.unpack_u4(d["w13_packed"])
    assert q.min() == 0 and q.max() == 15 and abs(q.mean() - 7.5) < 0.1
    s = workloads.bf16_bits_to_f32(d["w13_scale"])
    assert s.min() >= 0.0099 and s.max() <= 0.0301
    b = workloads.bf16_bits_to_f32(d["w13_bias"]).astype(np.float64)
    assert np.abs(b + 8 * s).max() < 0.006


# --------------------------------------------------------------------------- #
# mutation tests: each plants one mistake in the oracle; some pin must fail
# --------------------------------------------------------------------------- #
def _mutations():
    orig = {n: getattr(moe_ref, n) for n in
            ("unpack_u4", "dequant", "expert_swiglu_exact", "topk_route", "expert_down_exact",
             "expert_weights", "stable_permutation", "round_bf16", "block_map", "exclusive_scan",
             "router_logits", "rms_norm")}

    def msb_first(p):
        q = orig["unpack_u4"](p)
        return q.reshape(*q.shape[:-1], -1, 8)[..., ::-1].reshape(q.shape)

    def no_bias(packed, scale_bits, bias_bits):
        return orig["dequant"](packed, scale_bits, np.zeros_like(bias_bits))

    def silu_on_up(xrows, w13):
        F = w13.shape[0] // 2
        g, u = xrows @ w13[:F].T, xrows @ w13[F:].T
        return moe_ref.silu(u) * g

    def ties_high(logits, k):
        lg = np.asarray(logits, np.float32)
        ids, w = orig["topk_route"](lg[:, ::-1], k)
        return (lg.shape[1] - 1 - ids).astype(np.int32), w

    def no_renorm(logits, k):
        ids, w = orig["topk_route"](logits, k)
        lg = np.asarray(logits, np.float64)
        p = np.exp(lg - lg.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return ids, np.take_along_axis(p, ids.astype(np.int64), 1)

    def down_transposed(h, w2):
        return h @ w2 if h.shape[1] == w2.shape[0] else h @ w2.T * 1.0001

    def no_shared(wts, e):
        w13, w2 = orig["expert_weights"](wts, e)
        if e == wts["w13_packed"].shape[0] - 1:
            return w13 * 0, w2 * 0
        return w13, w2

    def unstable(ids):
        perm, inv = orig["stable_permutation"](ids)
        flat = np.asarray(ids).ravel()
        perm = perm.copy()
        for e in np.unique(flat):
            sel = np.nonzero(flat[perm] == e)[0]
            perm[sel] = perm[sel][::-1]
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.size, dtype=np.int32)
        return perm, inv

    def truncate(a):
        a = np.asarray(a, dtype=np.float64)
        m, e = np.frexp(a)
        return np.ldexp(np.trunc(m * 256.0), e - 8)

    def bm_no_shared(counts, offsets, T, block_n):
        bm = orig["block_map"](counts, offsets, T, block_n)
        return bm[bm[:, 0] < len(counts)]

    def inclusive(counts):
        c = np.asarray(counts, np.int64)
        return np.concatenate([np.cumsum(c), [c.sum()]]).astype(np.int32)

    def router_drops_last_k(x_bits, wr_bits):
        return orig["router_logits"](np.asarray(x_bits)[:, :-1], np.asarray(wr_bits)[:, :-1])

    def router_reversed_k(x_bits, wr_bits):
        return orig["router_logits"](np.asarray(x_bits)[:, ::-1], np.asarray(wr_bits))

    def rms_sum_not_mean(x_bits, eps=moe_ref.RMS_EPS):
        x = moe_ref.bf16_value(x_bits)
        return moe_ref.round_bf16(x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps))

    def scale_bias_swapped(packed, scale_bits, bias_bits):
        return orig["dequant"](packed, bias_bits, scale_bits)

    def sigmoid_for_silu(g):
        return 1.0 / (1.0 + np.exp(-g))

    def rms_eps_outside(x_bits, eps=moe_ref.RMS_EPS):
        x = moe_ref.bf16_value(x_bits)
        return moe_ref.round_bf16(x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps))

    def logits_rounded(x_bits, wr_bits):
        return moe_ref.round_bf16(orig["router_logits"](x_bits, wr_bits)).astype(np.float32)

    def tiles_too_tall(counts, offsets, T, block_n):
        return orig["block_map"](counts, offsets, T, block_n + 1)

    def nibble_pairs_swapped(p):
        q = orig["unpack_u4"](p)
        return q.reshape(*q.shape[:-1], -1, 2)[..., ::-1].reshape(q.shape)

    def groups_of_32(packed, scale_bits, bias_bits):
        q = orig["unpack_u4"](packed).astype(np.float64)
        K = q.shape[-1]
        s = np.repeat(moe_ref.bf16_value(scale_bits), 32, axis=-1)
        b = np.repeat(moe_ref.bf16_value(bias_bits), 32, axis=-1)
        s = np.concatenate([s, s], axis=-1)[..., :K]
        b = np.concatenate([b, b], axis=-1)[..., :K]
        return moe_ref.round_bf16(q * s + b)

    def ids_sorted_weights_not(logits, k):
        ids, w = orig["topk_route"](logits, k)
        return np.sort(ids, axis=1), w

    def signed_nibbles(p):
        return orig["unpack_u4"](p) - 8

    def perm_token_major(ids):
        n = np.asarray(ids).size
        perm = np.arange(n, dtype=np.int32)
        return perm, perm.copy()

    return {
        "topk_ids_sorted_weights_not": ("topk_route", ids_sorted_weights_not),
        "nibbles_signed": ("unpack_u4", signed_nibbles),
        "permutation_not_grouped_by_expert": ("stable_permutation", perm_token_major),
        "dequant_scale_bias_swapped": ("dequant", scale_bias_swapped),
        "silu_is_sigmoid": ("silu", sigmoid_for_silu),
        "rms_norm_eps_outside_sqrt": ("rms_norm", rms_eps_outside),
        "router_logits_rounded_to_bf16": ("router_logits", logits_rounded),
        "block_map_tiles_one_too_tall": ("block_map", tiles_too_tall),
        "nibble_pairs_swapped": ("unpack_u4", nibble_pairs_swapped),
        "dequant_groups_of_32": ("dequant", groups_of_32),
        "rms_norm_sum_not_mean": ("rms_norm", rms_sum_not_mean),
        "router_drops_last_k": ("router_logits", router_drops_last_k),
        "router_reversed_k": ("router_logits", router_reversed_k),
        "nibble_msb_first": ("unpack_u4", msb_first),
        "dequant_drops_bias": ("dequant", no_bias),
        "silu_on_up": ("expert_swiglu_exact", silu_on_up),
        "ties_to_high_index": ("topk_route", ties_high),
        "no_renormalisation": ("topk_route", no_renorm),
        "down_transposed": ("expert_down_exact", down_transposed),
        "y_not_rounded": ("down_output", lambda y: np.asarray(y, dtype=np.float64)),
        "shared_expert_dropped": ("expert_weights", no_shared),
        "unstable_scatter": ("stable_permutation", unstable),
        "bf16_truncation": ("round_bf16", truncate),
        "block_map_drops_shared": ("block_map", bm_no_shared),
        "inclusive_scan": ("exclusive_scan", inclusive),
    }


MUTATIONS = _mutations()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(moe_ref, attr, fn)
    failed = []
    checks = P.ALL_PINS + [lambda: P.pin_bruteforce_layer(shape=(128, 4, 2, 64), T=9, seed=1)]
    for pin in checks:
        try:
            pin()
        except AssertionError:
            failed.append(getattr(pin, "__name__", "brute"))
        except Exception as ex:  # a mutation that breaks shapes is caught too
            failed.append(f"{getattr(pin, '__name__', 'brute')}:{type(ex).__name__}")
    assert failed, f"mutation {name} slipped through every pin"
