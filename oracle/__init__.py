"""CPU oracle for the block-scaled FP4 path (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package; the product path never does.
"""
from .fp4_oracle import *  # noqa: F401,F403
from . import fp4_oracle  # noqa: F401
