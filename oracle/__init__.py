"""CPU oracle for the W4 mixture-of-experts FFN layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of what the layer computes, written
from the pages ("Perplexity Open Sources Lily" on aitrending.vip, the itinai.com
post on the Lily engine, and Labomaru's "Quick Take") and from the readings
listed in the repository's design notes where they are silent.  It shares no
code with the CUDA library and is imported only by the tests, by the smoke
check and by the benchmark's CPU-baseline leg.  The product path never calls it.

Modules:
  moe_ref         the vectorised oracle (per-expert grouping, float64 BLAS)
  brute           an independent per-token brute force used to pin moe_ref
  calibrate_skew  the script that fixed the skewed workload's bias scale

Pin status: routing, dequantisation, SwiGLU and the combine are pinned by the
brute force, by closed forms and by invariants (tests/test_oracle_pins.py).
No function of this package is "parity unpinned".
"""
