"""CPU oracle for the KDA layer core -- test infrastructure only.

A plain token-by-token fp64 recurrence (``kda_oracle.c``) plus its ctypes
front-end.  Only the tests, the smoke check and the benchmark's CPU-baseline
leg may import it; the CUDA library never does.
"""
from .oracle import Oracle, decode_step, default, gated_rmsnorm, prefill  # noqa: F401
