"""GB300-native (sm_103a) LiSA forward layer.

The compute lives in liblisa.so (hand-written CUDA kernels behind the C ABI
declared in include/lisa.h); ``lisa`` is its ctypes binding and ``build``
compiles it in-tree with nvcc.
"""
from . import lisa  # noqa: F401
from .lisa import LisaError, forward, load  # noqa: F401

__all__ = ["lisa", "forward", "load", "LisaError"]
