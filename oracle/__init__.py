"""The oracle: a plain, slow, float64 CPU implementation of what the CUDA path computes.

This package is TEST INFRASTRUCTURE.  Only the tests, the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  The library (``attention_fa2_forward_02_gb300``) never imports it and shares
no code with it; the only common module is the seeded input generator
(``attention_fa2_forward_02_gb300.synth``), which holds none of the method's
arithmetic and is called by the tests, not by the oracle.

Modules:

* :mod:`oracle.attention` - attention forward (O and the row log-sum-exp) and
  the analytic backward (dQ, dK, dV), as explicit score matrices in float64.
* :mod:`oracle.psa` - the PSA pack / extract / merge index maps and their
  adjoints, element-for-element.

Parity pins (tests/test_oracle.py, marked "not gpu"): brute-force evaluation on
tiny inputs, the worked examples the pages print, closed forms and invariants,
central finite differences for the gradients, and brute-force index loops for
the PSA maps.  Every function here is pinned; none is "parity unpinned".
"""
from . import attention, psa  # noqa: F401
