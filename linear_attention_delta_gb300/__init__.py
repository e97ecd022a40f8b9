"""GB300-native Kaczmarz Linear Attention: chunkwise forward and decode step.

The compute runs in the CUDA library ``libkla.so`` (sm_103a), reached through
its C ABI (``include/kla.h``) by the thin ctypes binding in ``kla.py``.  There
is no CPU fallback: calling into the library without it built, or without a
GPU, raises.
"""
from .kla import (KlaError, chunk_fwd, decode_step, load_library,  # noqa: F401
                  status_string)

__all__ = ["KlaError", "chunk_fwd", "decode_step", "load_library",
           "status_string"]
