"""PRISM mixer forward pass for GB300 (sm_103a): a C-ABI CUDA library
(``include/prism.h``, built into ``_build/libprism.so``) with a thin ctypes
binding (``prism``) and seeded synthetic inputs (``inputs``).

Submodules load lazily so that the input generator can be used without the
built library; every compute call goes through libprism.so and raises if it
is missing.
"""
__all__ = ["prism", "inputs", "build"]
