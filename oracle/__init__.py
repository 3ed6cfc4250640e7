"""fp64 CPU oracle for MLA latent-cache decode (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline legs import
this package. The CUDA library never does.
"""
from .mla_oracle import *  # noqa: F401,F403
