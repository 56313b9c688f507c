"""Brute-force per-token restatement of the layer, used only to pin ``moe_ref``.

Nothing here is vectorised across tokens or experts and nothing is shared with
``moe_ref``: nibbles are decoded with integer division, bf16 rounding works on
the float64 bit pattern, top-k is repeated selection, and each token visits its
own k experts plus the shared expert with no permutation or grouping.  It is
meant for tiny shapes only.
"""
from __future__ import annotations

import math
import struct

import numpy as np


def bf16_of_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def rne_bf16(v: float) -> float:
    """Round a float64 to bf16 (8 significant bits, float32's exponent range), ties to even, on
    its bit pattern: drop the float64 fraction bits bf16 does not keep -- 45 of 52 for normal
    results, more below 2**-126 where bf16's spacing stays 2**-133 -- and round on the rest."""
    if v == 0.0 or v != v or abs(v) == float("inf"):
        return v
    u = struct.unpack("<Q", struct.pack("<d", v))[0]
    sign = u >> 63
    exp = (u >> 52) & 0x7FF                  # biased float64 exponent of |v|
    drop = 52 - 7                             # fraction bits float64 keeps beyond bf16's 7
    mag = u & ((1 << 63) - 1)
    if exp - 1023 < -126:
        # bf16 subnormal: spacing 2**-133; a float64 |v| = mant * 2**(exp-1075) with the implicit
        # bit in mant, so the bits below 2**-133 are the lowest (-133) - (exp - 1075) of mant
        mant = (mag & ((1 << 52) - 1)) | (1 << 52)
        shift = (1075 - 133) - exp + 0        # bits of mant below the 2**-133 place
        if shift > 60:
            return -0.0 if sign else 0.0
        keep, rem, half = mant >> shift, mant & ((1 << shift) - 1), 1 << (shift - 1)
        if rem > half or (rem == half and (keep & 1)):
            keep += 1
        return (-1.0 if sign else 1.0) * keep * 2.0 ** -133
    keep = mag >> drop
    rem = mag & ((1 << drop) - 1)
    half = 1 << (drop - 1)
    if rem > half or (rem == half and (keep & 1)):
        keep += 1
    r = struct.unpack("<d", struct.pack("<Q", (keep << drop) | (sign << 63)))[0]
    if abs(r) > (2.0 - 2.0 ** -7) * 2.0 ** 127:
        return -float("inf") if sign else float("inf")
    return r


def nibble(word: int, i: int) -> int:
    return (int(word) // (16 ** i)) % 16


def dequant_row(words, scales, biases) -> list:
    """One weight row: element kk = 8*w + i uses group kk // 64."""
    out = []
    for w, word in enumerate(words):
        for i in range(8):
            kk = 8 * w + i
            s = bf16_of_bits(scales[kk // 64])
            b = bf16_of_bits(biases[kk // 64])
            out.append(rne_bf16(nibble(word, i) * s + b))
    return out


class ExpertCache:
    def __init__(self, wts):
        self.wts = wts
        self.cache = {}

    def get(self, e):
        if e not in self.cache:
            w = self.wts
            w13 = np.array([dequant_row(w["w13_packed"][e][r], w["w13_scale"][e][r], w["w13_bias"][e][r])
                            for r in range(w["w13_packed"].shape[1])])
            w2 = np.array([dequant_row(w["w2_packed"][e][r], w["w2_scale"][e][r], w["w2_bias"][e][r])
                           for r in range(w["w2_packed"].shape[1])])
            self.cache[e] = (w13, w2)
        return self.cache[e]


def topk_one(logits_row, k):
    """Pick the largest remaining logit k times; on equal logits the lower index wins."""
    vals = [float(v) for v in np.asarray(logits_row, dtype=np.float32)]
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(vals):
            if e in chosen:
                continue
            if best is None or v > vals[best]:
                best = e
        chosen.append(best)
    m = vals[chosen[0]]
    z = [math.exp(vals[e] - m) for e in chosen]
    s = sum(z)
    return chosen, [v / s for v in z]


def ffn_one(x, w13, w2):
    F = w13.shape[0] // 2
    h = []
    for f in range(F):
        g = float(np.dot(w13[f], x))
        u = float(np.dot(w13[F + f], x))
        h.append(rne_bf16(g / (1.0 + math.exp(-g)) * u))
    h = np.array(h)
    # the down projection's rows are bf16 as well
    return np.array([rne_bf16(float(np.dot(w2[c], h))) for c in range(w2.shape[0])]), h


def forward(x_bits, logits, wts, k):
    """Per token: out = bf16(sum_j w_j * FFN_{e_j}(x) + FFN_shared(x)), each FFN output row rounded to bf16."""
    T, E = np.asarray(logits).shape
    cache = ExpertCache(wts)
    outs, all_ids, all_w = [], [], []
    for t in range(T):
        x = np.array([bf16_of_bits(b) for b in x_bits[t]])
        ids, ws = topk_one(logits[t], k)
        total = None
        for e, wt in list(zip(ids, ws)) + [(E, 1.0)]:
            w13, w2 = cache.get(e)
            y, _ = ffn_one(x, w13, w2)
            total = wt * y if total is None else total + wt * y
        outs.append([rne_bf16(float(v)) for v in total])
        all_ids.append(ids)
        all_w.append(ws)
    return np.array(outs), np.array(all_ids, dtype=np.int32), np.array(all_w)
