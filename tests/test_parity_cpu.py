"""The layer parity checker (tests/parity.py) on the CPU: it accepts a float32
emulation of the GPU's arithmetic (FP32 accumulation, bf16 roundings of h and
y, FP32 combine), and it rejects planted mistakes in that emulation -- an h or
y value one bf16 step off where no accumulation error can explain it, a wrong
output element, a swapped row."""
import numpy as np
import pytest

import workloads
from oracle import moe_ref

import parity


def emulate_gpu(d, block_n=8):
    """The layer in float32 arithmetic laid out like the GPU's buffers (rows in expert order)."""
    wl = d["workload"]
    s = wl.shape
    T, H, E, k, F = wl.T, s.H, s.E, s.k, s.F
    A = T * k
    r = moe_ref.route(d["logits"], k, block_n)
    x = moe_ref.bf16_value(d["x_bits"]).astype(np.float32)
    h = np.zeros((A + T, F))
    y = np.zeros((A + T, H))
    for e in range(E + 1):
        rows = np.arange(A, A + T) if e == E else np.arange(r["offsets"][e], r["offsets"][e + 1])
        if rows.size == 0:
            continue
        toks = rows - A if e == E else r["perm"][rows] // k
        w13, w2 = moe_ref.expert_weights(d, e)
        g = x[toks] @ w13[:F].T.astype(np.float32)
        u = x[toks] @ w13[F:].T.astype(np.float32)
        hv = (g / (np.float32(1) + np.exp(-g))) * u
        h[rows] = moe_ref.round_bf16(hv.astype(np.float64))
        yv = h[rows].astype(np.float32) @ w2.T.astype(np.float32)
        y[rows] = moe_ref.round_bf16(yv.astype(np.float64))
    out = np.zeros((T, H), np.float32)
    wf = r["topk_w"].astype(np.float32)
    for j in range(k):
        out += wf[:, j:j + 1] * y[r["inv_perm"][np.arange(T) * k + j]].astype(np.float32)
    out += y[A:].astype(np.float32)
    return {"topk_ids": r["topk_ids"], "inv_perm": r["inv_perm"], "perm": r["perm"], "block_map": r["block_map"],
            "num_blocks": r["num_blocks"], "h": h, "y": y, "out": moe_ref.round_bf16(out.astype(np.float64))}


@pytest.fixture(scope="module")
def case():
    d = workloads.make_workload(workloads.custom(96, 256, 16, 4, 128), 3)
    return d, emulate_gpu(d)


def test_checker_accepts_float32_emulation(case):
    d, g = case
    st = parity.check_layer_arrays(d, g, what="float32 emulation")
    assert st["outputs"] == 96 * 256
    assert st["h_total"] == 96 * 5 * 128 and st["y_total"] == 96 * 5 * 256


def _exact_h(d, g, row):
    """Exact (float64) h of GPU row `row` and whether it is far from a rounding midpoint."""
    wl = d["workload"]
    T, k, E, F = wl.T, wl.shape.k, wl.shape.E, wl.shape.F
    A = T * k
    e = E if row >= A else int(g["topk_ids"].ravel()[g["perm"][row]])
    t = row - A if row >= A else int(g["perm"][row]) // k
    w13, _ = moe_ref.expert_weights(d, e)
    x = moe_ref.bf16_value(d["x_bits"][t])
    return moe_ref.expert_swiglu_exact(x[None], w13)[0], t


def _one_step(v, up=True):
    lo, hi = moe_ref.bf16_floor_ceil(np.nextafter(v, np.inf if up else -np.inf))
    return hi if up else lo


def test_checker_rejects_h_off_by_one_step(case):
    d, g = case
    g = {n: (v.copy() if isinstance(v, np.ndarray) else v) for n, v in g.items()}
    row = 5
    hx, t = _exact_h(d, g, row)
    lo, hi = moe_ref.bf16_floor_ceil(hx)
    frac = np.where(hi > lo, (hx - lo) / np.where(hi > lo, hi - lo, 1), 0.5)
    f = int(np.argmin(np.abs(frac - 0.1)))       # exact value close to the lower neighbour: no flip can reach hi
    g["h"][row, f] = _one_step(g["h"][row, f], up=True)
    with pytest.raises(AssertionError, match="h of token"):
        parity.check_layer_arrays(d, g, tokens=[t], what="planted h")


def test_checker_rejects_y_off_by_one_step(case):
    d, g = case
    g = {n: (v.copy() if isinstance(v, np.ndarray) else v) for n, v in g.items()}
    row = 7
    g["y"][row, 3] = _one_step(_one_step(g["y"][row, 3], up=True), up=True)
    t = int(g["perm"][row]) // d["workload"].shape.k
    with pytest.raises(AssertionError, match="y of token"):
        parity.check_layer_arrays(d, g, tokens=[t], what="planted y")


def test_checker_rejects_wrong_output(case):
    d, g = case
    g = {n: (v.copy() if isinstance(v, np.ndarray) else v) for n, v in g.items()}
    g["out"][11, 17] += 0.25 + 0.05 * abs(g["out"][11, 17])
    with pytest.raises(AssertionError, match="combine of the GPU's y"):
        parity.check_layer_arrays(d, g, what="planted out")


def test_checker_rejects_swapped_rows(case):
    d, g = case
    g = {n: (v.copy() if isinstance(v, np.ndarray) else v) for n, v in g.items()}
    g["h"][[2, 3]] = g["h"][[3, 2]]
    with pytest.raises(AssertionError, match="h of token"):
        parity.check_layer_arrays(d, g, what="swapped h rows")


def test_tile_tokens_cover_every_tile(case):
    d, g = case
    wl = d["workload"]
    toks = parity.tile_tokens(g["block_map"], g["num_blocks"], g["perm"], wl.T, wl.shape.k)
    A = wl.T * wl.shape.k
    inv = g["inv_perm"]
    rows = set()
    for t in toks:
        rows |= {int(inv[t * wl.shape.k + j]) for j in range(wl.shape.k)} | {A + int(t)}
    for e, r0, n in g["block_map"][:g["num_blocks"]]:
        assert (r0 + n - 1) in rows
