"""B300-native forward pass of a sparse Mixture-of-Experts FFN layer.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
``libmoe.so`` (declared in ``include/moe.h``); ``moe`` is its thin ctypes
binding.  Importing the package does not load the library: the first call
does, and raises if the library is missing.
"""

__all__ = ["moe", "synth"]
