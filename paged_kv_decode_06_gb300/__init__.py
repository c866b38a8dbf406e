"""GB300 (sm_103a) paged-KV decode attention.

The compute lives in the CUDA library ``libpagedattn.so`` (C ABI:
``include/paged_attn.h``); ``binding`` is its thin ctypes binding and
``workloads`` the seeded synthetic input generator.
"""
__version__ = "0.1.0"
