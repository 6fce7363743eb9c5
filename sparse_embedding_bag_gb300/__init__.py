"""GB300-native backward pass of pooled (EmbeddingBag) and unpooled embedding lookups
with a fused SGD / row-wise Adagrad update.

The computation lives in the CUDA library ``libembbwd.so`` (sources in ``csrc/``,
C ABI in ``include/embbwd.h``); ``embbwd`` is its thin ctypes binding, ``device``
moves seeded workloads (``synth``) to the GPU and calls the binding.
"""
__all__ = ["embbwd", "synth", "device", "build"]
