"""Independent fp64 CPU oracle for the LM-head log-prob library.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check in
``__graft_entry__`` and by the benchmark's CPU-baseline and reference legs.
The library (``invariant_lm_head_gb300``) never imports it and shares no code
with it.
"""

from .lmhead_oracle import *  # noqa: F401,F403
from . import loops  # noqa: F401
