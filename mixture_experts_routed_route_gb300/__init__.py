"""Dropless routed-expert MoE layer for one GB300 (sm_103a).

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/moe_gb300.h``); ``abi`` binds it with ctypes and ``layer`` wraps
it with torch-allocated buffers.  ``synth`` draws seeded synthetic
workloads.  Importing ``abi`` or ``layer`` fails if the library has not been
built: there is no CPU or eager fallback.
"""

__all__ = ["abi", "layer", "synth", "build"]
