"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin returns normally when the oracle agrees and raises AssertionError
otherwise, so the same functions serve the plain pin tests and the mutation
tests (which plant a mistake in the oracle and expect some pin to fail).
"""
from __future__ import annotations

import math
import os

import numpy as np

import workloads
from oracle import brute, moe_ref

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- #
# test-side helpers (independent of the oracle)
# --------------------------------------------------------------------------- #
def pack_q(q) -> np.ndarray:
    """Dense integers 0..15 [..., K] -> uint32 words [..., K/8], element 8w+i in bits [4i,4i+4)."""
    q = np.asarray(q, dtype=np.uint64)
    K = q.shape[-1]
    q = q.reshape(*q.shape[:-1], K // 8, 8)
    words = np.zeros(q.shape[:-1], dtype=np.uint64)
    for i in range(8):
        words |= q[..., i] << np.uint64(4 * i)
    return words.astype(np.uint32)


def bf16_bits(v: float) -> int:
    """bf16 bits of a float that is exactly representable in bf16."""
    u = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
    assert u & 0xFFFF == 0, v
    return u >> 16


def const_weights(E, rows13, H, rows2, F, q, s, b):
    def one(rows, K):
        return (pack_q(np.full((E + 1, rows, K), q)),
                np.full((E + 1, rows, K // 64), bf16_bits(s), np.uint16),
                np.full((E + 1, rows, K // 64), bf16_bits(b), np.uint16))
    p13, s13, b13 = one(rows13, H)
    p2, s2, b2 = one(rows2, F)
    return {"w13_packed": p13, "w13_scale": s13, "w13_bias": b13,
            "w2_packed": p2, "w2_scale": s2, "w2_bias": b2}


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return rows


# --------------------------------------------------------------------------- #
# pins
# --------------------------------------------------------------------------- #
def pin_round_bf16_library():
    """round_bf16 on float32-representable values equals torch's float32 -> bfloat16 (RNE)."""
    import torch
    r = np.random.default_rng(1)
    v = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-6, 6, 20000),
                        # exact ties: 9 significant bits with the last one set
                        (r.integers(256, 512, 4000) * 2 + 1) * 2.0 ** r.integers(-20, 20, 4000),
                        # the subnormal range (|v| < 2^-126, spacing 2^-133), ties there, and near the top
                        r.standard_normal(4000) * 2.0 ** r.integers(-149, -120, 4000),
                        (r.integers(0, 256, 1000) * 2 + 1) * 2.0 ** -134,
                        r.uniform(3.0e38, 3.4e38, 1000) * r.choice([-1, 1], 1000)]
                       ).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = moe_ref.round_bf16(v.astype(np.float64))
    assert np.array_equal(ref, got)


def pin_round_bf16_bitlevel():
    """round_bf16 on arbitrary float64 values equals the bit-level brute force (subnormals included)."""
    r = np.random.default_rng(2)
    v = np.concatenate([r.standard_normal(3000) * 10.0 ** r.integers(-5, 5, 3000),
                        r.standard_normal(1000) * 2.0 ** r.integers(-150, -118, 1000)])
    for a in v:
        assert moe_ref.round_bf16(np.array([a]))[0] == brute.rne_bf16(float(a)), a


def pin_dequant_golden():
    g = read_golden("dequant_cases.txt")
    for q, sb, bb, expect in (row for row in _rows_of(g)):
        packed = pack_q(np.array([[int(q)] + [0] * 63]))
        w = moe_ref.dequant(packed, np.array([[int(sb, 16)]], np.uint16), np.array([[int(bb, 16)]], np.uint16))
        assert w[0, 0] == float(expect), (q, sb, bb, w[0, 0], expect)


def _rows_of(g):
    # dequant_cases.txt lines have no key word: the parser used the q column as key
    for key, vals in g.items():
        for v in vals:
            yield [key] + v


def pin_dequant_exact_fraction():
    """Dequant equals an exact rational computation rounded to 8 significant bits."""
    from fractions import Fraction
    r = np.random.default_rng(3)
    q = r.integers(0, 16, size=(3, 128))
    sc = workloads.f32_to_bf16_bits(r.uniform(0.01, 0.03, size=(3, 2)).astype(np.float32))
    bi = workloads.f32_to_bf16_bits((r.uniform(-0.3, 0.3, size=(3, 2))).astype(np.float32))
    w = moe_ref.dequant(pack_q(q), sc, bi)

    def rne8(fr: Fraction) -> Fraction:
        if fr == 0:
            return fr
        sign = -1 if fr < 0 else 1
        a = abs(fr)
        e = 0
        while a >= 256:
            a /= 2
            e += 1
        while a < 128:
            a *= 2
            e -= 1
        fl = a.numerator // a.denominator
        rem = a - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        return sign * Fraction(fl) * Fraction(2) ** e

    for i in range(3):
        for kk in range(128):
            s = Fraction(float(workloads.bf16_bits_to_f32(sc[i, kk // 64])))
            b = Fraction(float(workloads.bf16_bits_to_f32(bi[i, kk // 64])))
            assert Fraction(float(w[i, kk])) == rne8(int(q[i, kk]) * s + b)


def pin_unpack_order():
    """Element 8w+i sits in bits [4i, 4i+4): 0x76543210 unpacks to 0..7."""
    got = moe_ref.unpack_u4(np.array([0x76543210, 0xFEDCBA98], dtype=np.uint32))
    assert list(got) == list(range(16))


def pin_routing_golden():
    g = read_golden("routing_tiny.txt")
    logits = np.array([[float(v) for v in row] for row in g["logits"]], dtype=np.float32)
    r = moe_ref.route(logits, 2, 2)
    assert r["topk_ids"].tolist() == [[int(v) for v in row] for row in g["ids"]]
    assert np.allclose(r["topk_w"], np.array([[float(v) for v in row] for row in g["w"]]), rtol=0, atol=1e-15)
    assert r["counts"].tolist() == [int(v) for v in g["counts"][0]]
    assert r["offsets"].tolist() == [int(v) for v in g["offsets"][0]]
    assert r["perm"].tolist() == [int(v) for v in g["perm"][0]]
    assert r["inv_perm"].tolist() == [int(v) for v in g["inv_perm"][0]]
    assert r["block_map"].tolist() == [[int(v) for v in row] for row in g["block"]]
    assert moe_ref.block_map_capacity(4, 6, 2, 2) == int(g["capacity"][0][0])


def pin_topk_bruteforce(T=200, E=16, k=4, seed=4):
    """topk_route equals repeated selection, including on rows with many ties."""
    r = np.random.default_rng(seed)
    lg = r.standard_normal((T, E)).astype(np.float32)
    lg[::3] = np.round(lg[::3])          # plenty of exact ties
    lg[5] = 0.0
    ids, w = moe_ref.topk_route(lg, k)
    for t in range(T):
        bi, bw = brute.topk_one(lg[t], k)
        assert ids[t].tolist() == bi
        assert np.allclose(w[t], bw, rtol=1e-14, atol=0)


def pin_topk_softmax_library(T=100, E=32, k=8, seed=5):
    """Renormalised top-k weights equal scipy's full softmax restricted to the chosen ids and
    renormalised; they sum to one."""
    from scipy.special import softmax
    r = np.random.default_rng(seed)
    lg = (3 * r.standard_normal((T, E))).astype(np.float32)
    ids, w = moe_ref.topk_route(lg, k)
    p = softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    # chosen logits are the k largest: every unchosen logit is <= the smallest chosen one
    for t in range(T):
        rest = np.setdiff1d(np.arange(E), ids[t])
        assert lg[t, rest].max() <= lg[t, ids[t]].min()


def check_routing_invariants(logits, k, block_n):
    T, E = logits.shape
    r = moe_ref.route(logits, k, block_n)
    ids, counts, offsets = r["topk_ids"], r["counts"], r["offsets"]
    perm, inv, bm = r["perm"], r["inv_perm"], r["block_map"]
    A = T * k
    assert counts.sum() == A
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    # textbook reductions
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert np.array_equal(np.sort(perm), np.arange(A))
    assert np.array_equal(perm[inv], np.arange(A))
    flat = ids.ravel()
    keys = flat[perm].astype(np.int64) * A + perm
    assert np.all(np.diff(keys) > 0)          # sorted by (expert, assignment): stable
    assert np.array_equal(np.bincount(perm // k, minlength=T), np.full(T, k))
    for e in range(E):
        assert np.all(flat[perm[offsets[e]:offsets[e + 1]]] == e)
    # the block map tiles [0, A + T) exactly, in order, one expert per tile
    nxt = 0
    for e_, r0, n in bm:
        assert r0 == nxt and 1 <= n <= block_n
        if e_ < E:
            assert offsets[e_] <= r0 and r0 + n <= offsets[e_ + 1]
        else:
            assert e_ == E and r0 >= A
        nxt = r0 + n
    assert nxt == A + T
    assert bm.shape[0] <= moe_ref.block_map_capacity(T, E, k, block_n)
    assert all(counts[e] == 0 or e in set(bm[:, 0].tolist()) for e in range(E))
    return r


def pin_routing_invariants():
    r = np.random.default_rng(6)
    for (T, E, k, bn) in ((1, 16, 2, 128), (37, 16, 2, 8), (300, 64, 8, 32), (64, 16, 16, 128)):
        check_routing_invariants(r.standard_normal((T, E)).astype(np.float32), k, bn)
    wl = workloads.WORKLOADS["prefill512"]
    tok = workloads.make_tokens(wl.shape, 512, 0)
    check_routing_invariants(tok["logits"], 8, 128)


def pin_closed_form_constant(T=5, H=128, E=4, k=2, F=64):
    """All q = 8, scale 2^-6, bias -2^-3 + 2^-5: every weight is 2^-5, so g = u = S/32 with
    S = sum_h x_h, h = bf16(silu(g) g), y_c = F h / 32 and out = bf16(2 y) (weights sum to 1,
    plus the shared expert)."""
    r = np.random.default_rng(7)
    x_bits = workloads.f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    logits = r.standard_normal((T, E)).astype(np.float32)
    wts = const_weights(E, 2 * F, H, H, F, 8, 2.0 ** -6, -2.0 ** -3 + 2.0 ** -5)
    out = moe_ref.moe_forward(x_bits, logits, wts, k)["out"]
    for t in range(T):
        S = float(workloads.bf16_bits_to_f32(x_bits[t]).astype(np.float64).sum())
        g = S / 32.0
        h = brute.rne_bf16(g / (1.0 + math.exp(-g)) * g)
        expect = brute.rne_bf16(2.0 * F * h / 32.0)
        assert np.all(out[t] == expect), (t, out[t][:4], expect)


def closed_form_perm_inputs(T=6, E=3, k=2, H=128, F=128, seed=8, down_scale=1.0):
    """Diagonal gate with per-group scales, up = c_e * identity, down = down_scale times a permutation."""
    assert H == F
    r = np.random.default_rng(seed)
    x_bits = workloads.f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    logits = r.standard_normal((T, E)).astype(np.float32)
    eye = np.eye(F, H, dtype=np.int64)
    up_c = [2, 3, 1, 5][: E + 1]
    g_scale = [[1.0, 0.5], [2.0, 0.25], [0.5, 4.0], [1.0, 1.0]][: E + 1]
    perms = [r.permutation(H) for _ in range(E + 1)]
    q13 = np.zeros((E + 1, 2 * F, H), np.int64)
    s13 = np.zeros((E + 1, 2 * F, H // 64), np.uint16)
    q2 = np.zeros((E + 1, H, F), np.int64)
    s2 = np.full((E + 1, H, F // 64), bf16_bits(down_scale), np.uint16)
    for e in range(E + 1):
        q13[e, :F] = eye
        q13[e, F:] = up_c[e] * eye
        for grp in range(H // 64):
            s13[e, :F, grp] = bf16_bits(g_scale[e][grp])
        s13[e, F:, :] = bf16_bits(1.0)
        q2[e, np.arange(H), perms[e]] = 1          # y_c = h_{perm[c]}
    wts = {"w13_packed": pack_q(q13), "w13_scale": s13, "w13_bias": np.zeros_like(s13),
           "w2_packed": pack_q(q2), "w2_scale": s2, "w2_bias": np.zeros_like(s2)}
    return x_bits, logits, wts, up_c, g_scale, perms


def pin_closed_form_permutation(T=6, E=3, k=2, H=128):
    """g_f = s_{e, f//64} x_f, u_f = c_e x_f, h = bf16(silu(g) u), y_c = h_{pi_e(c)};
    out = bf16(sum_j w_j y_{e_j} + y_shared) with w from the top-k logits."""
    x_bits, logits, wts, up_c, g_scale, perms = closed_form_perm_inputs(T, E, k, H, H)
    out = moe_ref.moe_forward(x_bits, logits, wts, k)["out"]
    for t in range(T):
        x = workloads.bf16_bits_to_f32(x_bits[t]).astype(np.float64)
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        z = [math.exp(float(logits[t, e]) - float(logits[t, order[0]])) for e in order]
        terms = [(e, zz / sum(z)) for e, zz in zip(order, z)] + [(E, 1.0)]
        for c in range(H):
            tot = 0.0
            for e, wt in terms:
                f = perms[e][c]
                g = g_scale[e][f // 64] * x[f]
                h = brute.rne_bf16(g / (1.0 + math.exp(-g)) * up_c[e] * x[f])
                tot += wt * h
            assert out[t, c] == brute.rne_bf16(tot), (t, c)


def pin_closed_form_scaled_down(T=6, E=3, k=2, H=128):
    """The permutation closed form with a down weight of 3 * 2^-7: y_c = bf16(3 * 2^-7 * h_{pi_e(c)})
    needs up to 10 significant bits before its rounding, so y is not bf16-exact and the rounding of
    the down projection's output to bf16 is pinned: out = bf16(sum_j w_j y_{e_j} + y_shared)."""
    a = 3.0 * 2.0 ** -7
    x_bits, logits, wts, up_c, g_scale, perms = closed_form_perm_inputs(T, E, k, H, H, down_scale=a)
    out = moe_ref.moe_forward(x_bits, logits, wts, k)["out"]
    inexact = 0
    for t in range(T):
        x = workloads.bf16_bits_to_f32(x_bits[t]).astype(np.float64)
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        z = [math.exp(float(logits[t, e]) - float(logits[t, order[0]])) for e in order]
        terms = [(e, zz / sum(z)) for e, zz in zip(order, z)] + [(E, 1.0)]
        for c in range(H):
            tot = 0.0
            for e, wt in terms:
                f = perms[e][c]
                g = g_scale[e][f // 64] * x[f]
                h = brute.rne_bf16(g / (1.0 + math.exp(-g)) * up_c[e] * x[f])
                y = brute.rne_bf16(a * h)
                inexact += y != a * h
                tot += wt * y
            assert out[t, c] == brute.rne_bf16(tot), (t, c)
    assert inexact > T * H  # most y values really are rounded


def pin_router_logits_integer(T=5, H=192, E=7, seed=12):
    """Router projection on small-integer operands (exact in bf16 and in float32): every logit equals
    the integer dot product x[t] . Wr[e], computed here with Python integers."""
    r = np.random.default_rng(seed)
    xi = r.integers(-3, 4, size=(T, H))
    wi = r.integers(-2, 3, size=(E, H))
    got = moe_ref.router_logits(workloads.f32_to_bf16_bits(xi.astype(np.float32)),
                                workloads.f32_to_bf16_bits(wi.astype(np.float32)))
    assert got.shape == (T, E) and got.dtype == np.float32
    for t in range(T):
        for e in range(E):
            assert got[t, e] == float(sum(int(a) * int(b) for a, b in zip(xi[t], wi[e]))), (t, e)


def pin_router_logits_exact_sum(T=3, H=128, E=5, seed=13):
    """Router projection on random bf16 operands: each logit is the exactly summed products
    (math.fsum) rounded once to float32."""
    r = np.random.default_rng(seed)
    xb = workloads.f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    wb = workloads.f32_to_bf16_bits((r.standard_normal((E, H)) / 11.0).astype(np.float32))
    got = moe_ref.router_logits(xb, wb)
    x = workloads.bf16_bits_to_f32(xb).astype(np.float64)
    w = workloads.bf16_bits_to_f32(wb).astype(np.float64)
    for t in range(T):
        for e in range(E):
            assert got[t, e] == np.float32(math.fsum(x[t] * w[e])), (t, e)


def pin_rms_norm(T=4, H=64, seed=14):
    """RMS norm: a constant row becomes all +-1 (up to eps, which bf16 cannot see); a constant row c
    whose square is comparable to eps (or below it) becomes c / sqrt(c^2 + 1e-6), the closed form that
    fixes where eps sits and its value (the reading of the layer's normalisation: eps = 1e-6 under
    the square root); and every output is the brute-force x / sqrt(mean x^2 + eps) rounded once to
    bf16."""
    const = np.array([[2.5] * H, [-0.375] * H], dtype=np.float32)
    got = moe_ref.rms_norm(workloads.f32_to_bf16_bits(const))
    assert np.array_equal(got, np.sign(const.astype(np.float64)))
    for c in (2.0 ** -10, -(2.0 ** -12)):
        got = moe_ref.rms_norm(workloads.f32_to_bf16_bits(np.full((1, H), c, dtype=np.float32)))
        want = brute.rne_bf16(c / math.sqrt(c * c + 1e-6))
        assert abs(want) < 0.75  # far from the +-1 of large rows: eps decides it
        assert np.all(got == want), (c, got[0, 0], want)
    r = np.random.default_rng(seed)
    xb = workloads.f32_to_bf16_bits((r.standard_normal((T, H)) * 3).astype(np.float32))
    got = moe_ref.rms_norm(xb)
    for t in range(T):
        row = [brute.bf16_of_bits(b) for b in xb[t]]
        scale = 1.0 / math.sqrt(math.fsum(v * v for v in row) / H + moe_ref.RMS_EPS)
        for c in range(H):
            assert got[t, c] == brute.rne_bf16(row[c] * scale), (t, c)


def pin_bruteforce_layer(shape=None, T=None, seed=0):
    """The vectorised oracle equals the per-token brute force on the tiny workload."""
    wl = workloads.WORKLOADS["tiny"] if shape is None else workloads.custom(T, *shape)
    d = workloads.make_workload(wl, seed)
    got = moe_ref.moe_forward(d["x_bits"], d["logits"], d, wl.shape.k)
    ref_out, ref_ids, ref_w = brute.forward(d["x_bits"], d["logits"], d, wl.shape.k)
    assert np.array_equal(got["topk_ids"], ref_ids)
    assert np.allclose(got["topk_w"], ref_w, rtol=1e-14, atol=0)
    assert np.array_equal(got["out"], ref_out)


ALL_PINS = [
    pin_round_bf16_library, pin_round_bf16_bitlevel, pin_dequant_golden, pin_dequant_exact_fraction,
    pin_unpack_order, pin_routing_golden, pin_topk_bruteforce, pin_topk_softmax_library,
    pin_routing_invariants, pin_closed_form_constant, pin_closed_form_permutation, pin_closed_form_scaled_down,
    pin_router_logits_integer, pin_router_logits_exact_sum, pin_rms_norm,
]
