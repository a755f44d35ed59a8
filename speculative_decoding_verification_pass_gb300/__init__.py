"""GB300-native speculative-decoding verification pass.

The compute path lives in a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/spec_verify.h``); ``binding`` is a
thin ctypes layer over it.  Importing this package does not load the library;
``binding.lib()`` does, and fails loudly when it has not been built.
"""
