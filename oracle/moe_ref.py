"""Float64 oracle of the W4 MoE FFN layer (test infrastructure only).

Step by step, in the pages' order:

1. router softmax + top-k: 8 of 256 experts per token ("Perplexity Open Sources
   Lily", Technical Details, Model bullet), the top-k softmax renormalised;
2. GPU-resident routing: per-expert histogram, exclusive prefix scan, scatter
   (a stable permutation of the assignments by expert) and block map (same
   page, Technical Details, Prefill optimizations bullet; Chinese section
   "预填充优化");
3. groupwise affine 4-bit weights, 64 weights per group with a bf16 scale (and
   bias, "affine"), expanded to bf16 only inside the grouped GEMM (same bullet;
   itinai.com post, paragraph 2: no full bfloat16 copy is allocated);
4. grouped SwiGLU expert GEMM with FP32 (here: exact float64) accumulation,
   whose outputs (h of the gate/up projection, y of the down projection) are
   bf16 rows in expert order;
5. weighted gather-combine of each token's k routed rows plus its shared-expert
   row (weight 1) back to token order (Technical Details, Model bullet: "8 of
   256 experts plus one shared expert").

Readings where the pages are silent (each is listed in the design notes):
ties in top-k go to the lower expert index; the dequantised weight is
round-to-nearest-even bf16 of the exact q*scale + bias; h = bf16(silu(g) * u);
y = bf16(h Wd^T) (the grouped GEMM writes bf16); the output is bf16 of the
exact weighted sum of the y rows.  Nibble k of a 32-bit word holds K element 8*w + k in bits
[4k, 4k+4).
"""
from __future__ import annotations

import numpy as np

GROUP = 64


# --------------------------------------------------------------------------- #
# number formats
# --------------------------------------------------------------------------- #
def bf16_value(bits) -> np.ndarray:
    """Exact float64 value of bf16 bit patterns (bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits and float32's exponent range.  With
    a = m * 2**e, 0.5 <= |m| < 1, a normal result (|a| >= 2**-126) is
    rint(m * 2**8) * 2**(e-8); below 2**-126 the spacing stays 2**-133 (the
    subnormals), so tiny values round to a multiple of it (possibly to a signed
    zero).  Values past the largest finite bf16 round to infinity.  numpy's rint
    rounds half to even.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    q = np.where(e >= -125, e - 8, -133)         # exponent of the spacing at a
    r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, a), r)


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def unpack_u4(packed) -> np.ndarray:
    """uint32 words [..., K/8] -> integers 0..15 [..., K]; element 8w+i in bits [4i, 4i+4)."""
    p = np.asarray(packed, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (p[..., :, None] >> shifts) & np.uint32(0xF)
    return q.reshape(*p.shape[:-1], p.shape[-1] * 8).astype(np.int64)


def dequant(packed, scale_bits, bias_bits) -> np.ndarray:
    """Groupwise affine 4-bit dequantisation: w = bf16(q * scale + bias), 64 weights per group.

    q*scale + bias is exact in float64 (a 4-bit integer times an 8-bit
    significand plus an 8-bit significand), so one rounding to bf16 gives the
    expanded weight the grouped GEMM multiplies with.
    """
    q = unpack_u4(packed).astype(np.float64)
    s = np.repeat(bf16_value(scale_bits), GROUP, axis=-1)
    b = np.repeat(bf16_value(bias_bits), GROUP, axis=-1)
    return round_bf16(q * s + b)


# --------------------------------------------------------------------------- #
# between layers
# --------------------------------------------------------------------------- #
RMS_EPS = 1e-6


def rms_norm(x_bits, eps: float = RMS_EPS) -> np.ndarray:
    """Unit-gain RMS norm of each token, the input of a layer in a stack of layers:
    bf16(x / sqrt(mean(x^2) + eps)), computed in float64 and rounded once.  The pages do
    not describe the model's normalisation; this is the plainest one."""
    x = bf16_value(x_bits)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return round_bf16(x * r)


# --------------------------------------------------------------------------- #
# router projection
# --------------------------------------------------------------------------- #
def router_logits(x_bits, wr_bits) -> np.ndarray:
    """Router projection: logits[t, e] = sum_h x[t, h] * Wr[e, h], rounded once to float32.

    The router chooses experts from one logit per expert ("Perplexity Open
    Sources Lily", Technical Details, Model bullet); here the logit is the dot
    product of the token's bf16 activations with the expert's bf16 router row.
    The products are exact in float64 and their float64 sum is within 1e-12
    relative of the exact sum, far inside the final float32 rounding.
    """
    x = bf16_value(x_bits)
    w = bf16_value(wr_bits)
    return (x @ w.T).astype(np.float32)


# --------------------------------------------------------------------------- #
# routing
# --------------------------------------------------------------------------- #
def topk_route(logits, k: int):
    """Router softmax + top-k, renormalised over the k chosen experts.

    Experts are ordered by descending logit, ties by ascending index; the first
    k are taken.  The weights softmax(l)[top] / sum(softmax(l)[top]) equal
    exp(l_j - l_max) / sum_{i in top} exp(l_i - l_max), computed in float64.
    Returns ids int32 [T, k] (in that order) and w float64 [T, k].
    """
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t]))
        ids[t] = order[:k]
    top = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    z = np.exp(top - top[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return ids, w


def histogram(ids, E: int) -> np.ndarray:
    """Per-expert count of assignments."""
    return np.bincount(np.asarray(ids).ravel(), minlength=E).astype(np.int32)


def exclusive_scan(counts) -> np.ndarray:
    """offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]; length E+1."""
    c = np.asarray(counts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(c)]).astype(np.int32)


def stable_permutation(ids):
    """Scatter: the assignments a = t*k + j sorted by (expert, a).

    perm[p] = a, inv_perm[a] = p.  Returns (perm, inv_perm), int32.
    """
    flat = np.asarray(ids).ravel()
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return perm, inv


def block_map(counts, offsets, T: int, block_n: int) -> np.ndarray:
    """Tile block map: for each expert e in ascending order and each tile i of
    block_n rows, (e, offsets[e] + i*block_n, min(block_n, counts[e] - i*block_n)).
    Experts with no assignment get no tile.  The shared expert follows as
    segment E over rows A .. A+T-1 (token t at row A + t).  int32 [nb, 3].
    """
    E = len(counts)
    A = int(offsets[E])
    rows = []
    for e in range(E):
        c = int(counts[e])
        for i in range(0, c, block_n):
            rows.append((e, int(offsets[e]) + i, min(block_n, c - i)))
    for i in range(0, T, block_n):
        rows.append((E, A + i, min(block_n, T - i)))
    return np.asarray(rows, dtype=np.int32).reshape(-1, 3)


def block_map_capacity(T: int, E: int, k: int, block_n: int) -> int:
    """Upper bound on the number of tiles: ceil(T*k/bn) + E + ceil(T/bn)."""
    A = T * k
    return -(-A // block_n) + E + -(-T // block_n)


def route(logits, k: int, block_n: int) -> dict:
    """All routing outputs for one layer call."""
    ids, w = topk_route(logits, k)
    T, E = np.asarray(logits).shape
    counts = histogram(ids, E)
    offsets = exclusive_scan(counts)
    perm, inv = stable_permutation(ids)
    bm = block_map(counts, offsets, T, block_n)
    return {"topk_ids": ids, "topk_w": w, "counts": counts, "offsets": offsets,
            "perm": perm, "inv_perm": inv, "block_map": bm, "num_blocks": bm.shape[0]}


# --------------------------------------------------------------------------- #
# expert FFN and combine
# --------------------------------------------------------------------------- #
def silu(g):
    return g / (1.0 + np.exp(-g))


def expert_swiglu_exact(xrows, w13) -> np.ndarray:
    """silu(x Wg^T) * (x Wu^T) before rounding; w13 holds the F gate rows then the F up rows."""
    F = w13.shape[0] // 2
    g = xrows @ w13[:F].T
    u = xrows @ w13[F:].T
    return silu(g) * u


def expert_swiglu(xrows, w13) -> np.ndarray:
    """h = bf16(silu(x Wg^T) * (x Wu^T))."""
    return round_bf16(expert_swiglu_exact(xrows, w13))


def bf16_floor_ceil(a):
    """The two bf16 values enclosing a (equal when a is a bf16 value), subnormals included."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    q = np.where(e >= -125, e - 8, -133)
    return np.ldexp(np.floor(np.ldexp(a, -q)), q), np.ldexp(np.ceil(np.ldexp(a, -q)), q)


def expert_down_exact(h, w2) -> np.ndarray:
    """h Wd^T, exact (float64), before the grouped GEMM's bf16 output rounding."""
    return h @ w2.T


def down_output(y_exact) -> np.ndarray:
    """y = bf16(h Wd^T): the down projection's rows are written as bf16 like h."""
    return round_bf16(y_exact)


def expert_weights(wts: dict, e: int):
    w13 = dequant(wts["w13_packed"][e], wts["w13_scale"][e], wts["w13_bias"][e])
    w2 = dequant(wts["w2_packed"][e], wts["w2_scale"][e], wts["w2_bias"][e])
    return w13, w2


def moe_forward(x_bits, logits, wts: dict, k: int, tokens=None, want_h: bool = False,
                want_y: bool = False) -> dict:
    """The layer: out[t] = bf16( sum_j w[t,j] * y_{e_j}(x_t) + y_shared(x_t) ), y = bf16(h Wd^T).

    ``tokens`` restricts the computation to a subset of token indices (routing
    of a token depends on its own logits only), which is how full-size
    workloads are checked on sampled outputs.  With ``want_h`` the bf16
    intermediate h of every (token, routed expert) and of the shared expert is
    returned as well, keyed by (t, e), together with its unrounded value
    (key "h_exact"); ``want_y`` does the same for the bf16 rows y of the down
    projection (keys "y" and "y_exact").
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    ids, w = topk_route(logits[sel], k)
    x = bf16_value(np.asarray(x_bits)[sel])
    n, H = x.shape
    acc = np.zeros((n, H), dtype=np.float64)
    hs, hx, ys, yx = {}, {}, {}, {}
    for e in sorted(set(np.unique(ids).tolist()) | {E}):
        if e == E:
            rows, wt = np.arange(n), np.ones(n)
        else:
            rows, cols = np.nonzero(ids == e)
            wt = w[rows, cols]
        w13, w2 = expert_weights(wts, e)
        v = expert_swiglu_exact(x[rows], w13)
        h = round_bf16(v)
        yv = expert_down_exact(h, w2)
        y = down_output(yv)
        for i, r in enumerate(rows):
            key = (int(sel[r]), int(e))
            if want_h:
                hs[key], hx[key] = h[i], v[i]
            if want_y:
                ys[key], yx[key] = y[i], yv[i]
        acc[rows] += wt[:, None] * y
    res = {"out": round_bf16(acc), "topk_ids": ids, "topk_w": w, "tokens": sel}
    if want_h:
        res["h"] = hs
        res["h_exact"] = hx
    if want_y:
        res["y"] = ys
        res["y_exact"] = yx
    return res
