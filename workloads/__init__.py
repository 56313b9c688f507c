"""Seeded synthetic inputs for the W4 mixture-of-experts FFN layer.

This module only draws random data and lays it out in the canonical formats; it
holds none of the layer's arithmetic (no top-k, no dequantisation, no GEMM).
Both the CPU oracle and the CUDA path consume exactly these arrays, so a parity
test compares the two on identical bits.

Workload shapes follow the pages' model description (a router choosing 8 of 256
experts plus one always-on shared expert; "Perplexity Open Sources Lily",
Technical Details, Model bullet) and their prefill prompt lengths (512-token
prompt, 4K prompt; same page, Benchmarks bullet; itinai.com post, paragraph 2).
The pages publish no tensors, so every value here is drawn from a fixed seed.

Canonical layouts (all row-major, little-endian):

* ``x_bits``      uint16 [T, H]       bf16 bit patterns of the activations.
* ``logits``      float32 [T, E]      router logits.
* ``w13_packed``  uint32 [E+1, 2F, H/8]  gate rows 0..F-1 then up rows F..2F-1;
  K element ``8*w + i`` sits in bits ``[4i, 4i+4)`` of word ``w``.
* ``w13_scale``, ``w13_bias``  uint16 [E+1, 2F, H/64]  bf16 bits, one pair per
  64 consecutive K ("64 weights per group", groupwise affine).
* ``w2_packed``   uint32 [E+1, H, F/8], ``w2_scale``/``w2_bias`` uint16 [E+1, H, F/64].
* Expert index ``E`` (the last) is the shared expert.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GROUP = 64  # weights per quantisation group


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Sizes of one MoE FFN layer: hidden H, routed experts E, top-k, expert width F."""

    H: int
    E: int
    k: int
    F: int


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    shape: LayerShape
    skew: bool = False
    desc: str = ""


TINY = LayerShape(H=256, E=16, k=2, F=128)
FULL = LayerShape(H=2048, E=256, k=8, F=512)

WORKLOADS = {
    "tiny": Workload("tiny", 64, TINY, desc="T=64, H=256, 16 experts top-2 + shared, F=128"),
    "prefill512": Workload("prefill512", 512, FULL, desc="T=512, H=2048, 256 experts top-8 + shared, F=512"),
    "prefill4k": Workload("prefill4k", 4096, FULL, desc="T=4096, same layer as prefill512"),
    "decode1": Workload("decode1", 1, FULL, desc="T=1 batch-1 decode, same layer"),
    "decode8": Workload("decode8", 8, FULL, desc="T=8 decode, same layer"),
    "skew16k": Workload("skew16k", 16384, FULL, skew=True,
                        desc="T=16384, same layer, Zipf(s=1.2) expert bias on the logits"),
}

# Zipf exponent of the per-expert logit offset of the skewed workload.
ZIPF_S = 1.2
# Scale of that offset.  Fixed once by bisection so that about 30 of the 256
# experts receive no assignment at T=16384 (oracle/calibrate_skew.py writes it).
SKEW_BETA = 0.869140625


# --------------------------------------------------------------------------- #
# bf16 <-> float32 bit conversion (storage format only)
# --------------------------------------------------------------------------- #
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- #
# generators
# --------------------------------------------------------------------------- #
def _rng(seed: int, *tag: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, *tag]))


def make_weights(shape: LayerShape, seed: int = 0) -> dict:
    """Packed uint4 expert weights with bf16 scale ~U(0.01,0.03) and bias -8*scale + N(0,1e-3).

    Every nibble of a uniformly random 32-bit word is an independent uniform
    integer in 0..15, so the packed words are drawn directly.
    """
    H, E, F = shape.H, shape.E, shape.F
    assert H % GROUP == 0 and F % GROUP == 0
    out = {}
    for tag, (rows, K) in ((13, (2 * F, H)), (2, (H, F))):
        r = _rng(seed, 1, tag, H, E, F)
        packed = r.integers(0, 2**32, size=(E + 1, rows, K // 8), dtype=np.uint32)
        scale = r.uniform(0.01, 0.03, size=(E + 1, rows, K // GROUP)).astype(np.float32)
        scale_bits = f32_to_bf16_bits(scale)
        scale_v = bf16_bits_to_f32(scale_bits).astype(np.float64)
        bias = -8.0 * scale_v + r.normal(0.0, 1e-3, size=scale_v.shape)
        bias_bits = f32_to_bf16_bits(bias.astype(np.float32))
        name = "w13" if tag == 13 else "w2"
        out[f"{name}_packed"] = packed
        out[f"{name}_scale"] = scale_bits
        out[f"{name}_bias"] = bias_bits
    return out


def router_weight(shape: LayerShape, seed: int = 0) -> np.ndarray:
    """Router projection W_r [E, H], fp32 ~N(0, sigma=1/sqrt(H)) so logits have sigma ~ 1."""
    r = _rng(seed, 2, shape.H, shape.E)
    return r.normal(0.0, 1.0 / math.sqrt(shape.H), size=(shape.E, shape.H)).astype(np.float32)


def router_weight_bits(shape: LayerShape, seed: int = 0) -> np.ndarray:
    """The router projection as bf16 bits [E, H] (the fp32 weight above, rounded): the operand of the
    fused router projection, which multiplies bf16 activations by bf16 router rows."""
    return f32_to_bf16_bits(router_weight(shape, seed))


def skew_offsets(E: int, beta: float = SKEW_BETA, seed: int = 0) -> np.ndarray:
    """Per-expert logit offset beta * (-s * ln rank_e), ranks a seeded permutation of 1..E."""
    r = _rng(seed, 3, E)
    rank = r.permutation(E) + 1
    return (beta * (-ZIPF_S * np.log(rank.astype(np.float64)))).astype(np.float32)


def make_tokens(shape: LayerShape, T: int, seed: int = 0, skew: bool = False,
                beta: float | None = None) -> dict:
    """Activations x ~N(0,1) as bf16 and router logits fp32(x . W_r^T) (+ the Zipf offset)."""
    r = _rng(seed, 4, T, shape.H, shape.E)
    x = r.standard_normal((T, shape.H), dtype=np.float32)
    x_bits = f32_to_bf16_bits(x)
    xv = bf16_bits_to_f32(x_bits).astype(np.float64)
    wr = router_weight(shape, seed).astype(np.float64)
    logits = (xv @ wr.T).astype(np.float32)
    if skew:
        logits = logits + skew_offsets(shape.E, SKEW_BETA if beta is None else beta, seed)[None, :]
        logits = logits.astype(np.float32)
    return {"x_bits": x_bits, "logits": logits}


def make_workload(name_or_wl, seed: int = 0, with_weights: bool = True) -> dict:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    d = {"workload": wl}
    d.update(make_tokens(wl.shape, wl.T, seed, wl.skew))
    if with_weights:
        d.update(make_weights(wl.shape, seed))
    return d


def custom(T: int, H: int, E: int, k: int, F: int, skew: bool = False) -> Workload:
    """An ad-hoc workload (parity tests use several small ragged shapes)."""
    return Workload(f"T{T}_H{H}_E{E}_k{k}_F{F}", T, LayerShape(H, E, k, F), skew)
