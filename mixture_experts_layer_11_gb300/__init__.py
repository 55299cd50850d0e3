"""GB300-native (sm_103a) Mixture-of-Experts layer: forward and backward.

The layer's steps run in hand-written CUDA kernels behind a C-ABI library
(``include/moe.h``); ``ops`` is its thin ctypes binding with the same entry
point names and ``layer`` composes them into one forward + backward pass.
Importing this package loads nothing native; the first call into ``ops``
loads the library and raises if it has not been built.
"""
__all__ = ["synth", "ops", "layer"]
