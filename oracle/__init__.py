"""CPU oracle for the fused 8-bit blockwise AdamW + stochastic-rounding step.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  See q8_oracle.c for
the readings it implements and the sources it follows.
"""
from .q8_oracle import *  # noqa: F401,F403
