"""GB300-native Kimi Delta Attention (KDA) layer core.

The compute lives in ``libkda.so`` (hand-written CUDA for sm_103a behind a C
ABI, see ``include/kda.h``); :mod:`.kda` is the thin ctypes binding with the
same entry-point names, and :mod:`.inputs` draws the seeded synthetic
workloads.  Importing the package does not load the library; the first call
through :mod:`.kda` does, and fails loudly if it has not been built.
"""
__all__ = ["kda", "inputs"]
