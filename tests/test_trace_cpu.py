"""The trace CLI's decoding of the trace words (bit_mixture_experts_gb300/trace.py), on synthetic
words laid out as moe_trace_read returns them: per CTA and warp, cycles waited, waits, the complement
of the first wait's start, the last wait's end."""
import numpy as np

from bit_mixture_experts_gb300.trace import ROLES, TRACE_CTAS, role_stats


def _words():
    return np.zeros((TRACE_CTAS, 32, 4), np.uint64)


def _slot(w, cta, warp, waited, waits, first, last):
    w[cta, warp] = [waited, waits, ~np.uint64(first), last]


def test_shares_spans_and_complement_encoding():
    w = _words()
    for cta, base in ((0, 10_000), (1, 2_000_000_000)):  # clock64 values far apart on two SMs
        _slot(w, cta, 0, 300, 3, base, base + 1000)               # producer waits 30%
        _slot(w, cta, 1, 100, 10, base + 100, base + 1100)        # MMA issuer waits 10%
        _slot(w, cta, 2, 500, 5, base, base + 1000)               # activation loads: one busy warp,
        for warp in range(4, 12):                                 # the other idle
            _slot(w, cta, warp, 200 + 100 * (warp % 2), 4, base, base + 1000)
        for warp in range(12, 16):
            _slot(w, cta, warp, 900, 2, base + 50, base + 1050)
    st = role_stats(w.reshape(-1), 2)
    assert set(st) == {name for name, _ in ROLES}
    assert abs(st["weight producer"]["wait_share_median"] - 0.3) < 1e-12
    assert abs(st["MMA issuer"]["wait_share_median"] - 0.1) < 1e-12
    # the role's span and both its warps: 500 cycles waited of 2 x 1000
    assert abs(st["activation loads"]["wait_share_median"] - 0.25) < 1e-12
    assert abs(st["dequantisation"]["wait_share_median"] - 0.25) < 1e-12
    assert abs(st["epilogue"]["wait_share_median"] - 0.9) < 1e-12
    assert st["epilogue"]["span_kcycles_max"] == 1.0
    assert st["dequantisation"]["waits_per_warp"] == 4
    assert all(r["ctas"] == 2 for r in st.values())


def test_idle_ctas_and_roles_are_left_out():
    w = _words()
    _slot(w, 0, 1, 10, 1, 5, 105)
    st = role_stats(w.reshape(-1), 4)  # CTAs 1-3 and every other role recorded nothing
    assert list(st) == ["MMA issuer"]
    assert st["MMA issuer"]["ctas"] == 1
    assert abs(st["MMA issuer"]["wait_share_median"] - 0.1) < 1e-12
