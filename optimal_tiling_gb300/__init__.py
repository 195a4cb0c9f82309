"""GB300-native exact softmax attention: fused streaming forward, recompute
backward and a materialising comparison variant, all as hand-written sm_103a
kernels behind a C ABI (``include/attn.h``).

Importing the package loads nothing; the CUDA library is loaded on the first
call through :mod:`optimal_tiling_gb300.attn` and a missing library is an error.
"""
__all__ = ["attn", "inputs", "iomodel"]
