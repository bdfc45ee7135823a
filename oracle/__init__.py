"""CPU oracle for the batch-1 decode step — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The engine (``autoregressive_decode_gb300``)
never imports it and shares no code, table or helper with it; the only shared
module is ``synthetic`` (seeded random inputs, no arithmetic of the method).

Precision: fp32, as the decode-engine specification fixes ("a plain, slow fp32
CPU implementation of the same decoder").

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
values the pages print, closed forms, invariants or brute force
(tests/test_oracle_pins.py).  No function is unpinned.
"""
from .oracle import *  # noqa: F401,F403
