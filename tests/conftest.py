import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the layer parity statistics gathered by the GPU tests (tests/gpu_util.py), so that a
    run's log records the plain-oracle miss counts and the rounding flips behind them."""
    try:
        import gpu_util
    except Exception:
        return
    stats = getattr(gpu_util, "PARITY_STATS", [])
    if not stats:
        return
    import parity
    tr = terminalreporter
    tr.write_sep("-", "layer parity statistics (tests/parity.py)")
    tot = {"outputs": 0, "misses_plain": 0, "miss_tokens": 0, "flip_tokens": 0, "tokens": 0, "misses_if_y_fp32": 0}
    for what, st in stats:
        tr.write_line(parity.summary_line(what, st))
        for key in tot:
            tot[key] += st[key]
    tr.write_line(f"parity total over {len(stats)} layer checks: {tot['outputs']} outputs, {tot['misses_plain']} "
                  f"outside 1e-2 + 1e-2|ref| of the plain oracle in {tot['miss_tokens']} tokens, every one of them "
                  f"a token with a validated h/y rounding flip ({tot['flip_tokens']} of {tot['tokens']} tokens have "
                  f"one); {tot['misses_if_y_fp32']} would remain if y were kept in FP32")
