"""GB300-native DSA (DeepSeek-style sparse attention) decode hot path.

The compute path is the CUDA library ``libdsa.so`` (hand-written sm_103a
kernels behind a C ABI declared in ``include/dsa.h``); ``binding`` marshals
torch tensors to it.  ``synth`` generates seeded synthetic workloads.
"""
__all__ = ["binding", "synth"]
