"""GB300-native hybrid sliding-window two-pool KV attention.

The compute path is the C-ABI library ``libswa`` (hand-written sm_103a CUDA,
declared in ``include/swa.h``); ``hybrid_sliding_window_gb300.api`` is its
thin ctypes binding.  Importing this package does not load the library;
the first call into ``api`` does, and raises if it is missing.
"""
__all__ = ["api", "synth"]
