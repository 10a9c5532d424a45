"""GB300-native batched acceptance step of a speculative-decoding verifier (SDCP).

``sdcp``: the binding of libsdcp (the CUDA C ABI declared in include/sdcp.h).
``synth``: seeded synthetic verify batches.  ``build_ext``: builds libsdcp.so with nvcc.
"""
__all__ = ["sdcp", "synth", "build_ext"]
