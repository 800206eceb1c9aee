"""fp64 CPU oracle of the sparse MoE layer -- test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import it. The CUDA library never calls it.
"""
from .moe_oracle import *  # noqa: F401,F403
