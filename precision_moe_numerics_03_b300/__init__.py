"""4-bit MoE expert-layer numerics for B300 (sm_103a).

The compute lives in the CUDA library ``libmoe4.so`` (``csrc/``) behind the C ABI declared in
``include/moe4.h``; ``moe4`` is the thin ctypes binding with the same entry-point names.  Importing
this package loads nothing; ``moe4.load()`` opens the library and raises if it is missing.
"""
__all__ = ["inputs", "moe4"]
