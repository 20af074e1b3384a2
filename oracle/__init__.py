"""Float64 CPU oracle for the INT4 decode block (test infrastructure only).

Only the test-suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA path.
"""
from .futr_oracle import *  # noqa: F401,F403
from . import futr_oracle  # noqa: F401
