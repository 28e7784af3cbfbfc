"""GB300-native (sm_103a) weight-only 4-bit fused Mixture-of-Experts layer.

The compute lives in a C-ABI CUDA library (``include/moe_w4a16.h``); ``binding``
is its thin ctypes binding and ``layer`` a convenience wrapper that allocates
the buffers with PyTorch.  Importing this package does not load the library.
"""
