"""fp64 CPU oracle of the hybrid attention layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never uses it.
"""
from .oracle import *  # noqa: F401,F403
