"""GB300-native (sm_103a) smoothed INT8/FP8 quantized attention.

The compute lives in libsage.so (include/sage.h); ``sage`` is its thin ctypes
binding and ``workloads`` the seeded synthetic inputs.  Import ``sage``
explicitly: it loads (and if needed builds) the CUDA library.
"""
__all__ = ["sage", "workloads"]
