"""GB300-native grouped scaled activation fused with MXFP8/NVFP4 quantization.

The compute path is the CUDA library ``libgsa.so`` (C ABI in include/gsa.h),
reached through the ctypes binding in :mod:`.gsa`.  :mod:`.inputs` draws the
seeded synthetic workloads.
"""
__all__ = ["gsa", "inputs", "build"]
