"""GB300-native error-feedback gradient compressor.

The compressor runs in the CUDA library ``libgc.so`` behind the C ABI of
``include/gc.h``; ``gradient_compression_ef_gb300.gc`` is the thin ctypes
binding to it and ``gradient_compression_ef_gb300.inputs`` draws the seeded
synthetic workloads.  Importing this package loads nothing native.
"""
__all__ = ["gc", "inputs"]
