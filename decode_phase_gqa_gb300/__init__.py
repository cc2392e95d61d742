"""GB300-native decode-phase GQA attention over a paged KV cache.

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/kvattn.h``); ``kvattn`` is its thin
ctypes binding.  ``workloads`` draws seeded synthetic inputs.
"""
