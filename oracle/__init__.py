"""CPU oracle for the single-GPU MoE layer (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. The product library never calls it and shares no code with it.
"""
from .moe_oracle import *  # noqa: F401,F403
