"""The trace build's wait statistics on the GPU: `python -m bit_mixture_experts_gb300.trace` (run as its
own process, since it loads libmoe_w4_trace.so in place of the product library) traces the kernels of a
full-size workload; the warps of every role report waits on every CTA and the shares lie in [0, 1]."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,kernels", [("prefill512", 1), ("prefill4k", 2)])
def test_trace_cli(workload, kernels):
    r = subprocess.run([sys.executable, "-m", "bit_mixture_experts_gb300.trace", "--workload", workload, "--json"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    rep = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(rep["kernels"]) == kernels
    for name, k in rep["kernels"].items():
        roles = k["roles"]
        assert set(roles) == {"weight producer", "MMA issuer", "activation loads", "dequantisation", "epilogue"}, name
        for role, st in roles.items():
            assert st["ctas"] == rep["ctas"], (name, role)
            assert 0.0 <= st["wait_share_min"] <= st["wait_share_median"] <= st["wait_share_max"] <= 1.0, (name, role)
            assert st["waits_per_warp"] >= 1, (name, role)
        assert k["us"] > 0, name
