"""Context-parallel attention primitives for B300 (sm_103a).

The compute lives in the CUDA library ``libcpattn.so`` (C ABI: ``include/cpattn.h``); the Python
binding is ``context_math_non_b300.cpattn``.  Importing the package does not load the library,
so the seeded workload drawer (``context_math_non_b300.inputs``) is usable without a GPU; the
first binding call loads it and fails loudly if it is missing.
"""
__version__ = "0.1.0"
