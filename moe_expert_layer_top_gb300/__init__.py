"""GB300-native small-batch MXFP8 MoE step.

The compute path is the C-ABI library ``libmoe.so`` (hand-written sm_103a CUDA
kernels, declared in include/moe.h). ``abi`` is its thin ctypes binding, and
``layer`` wraps it for PyTorch device memory and streams. ``build.build()``
compiles the library in-tree.
"""
from . import abi, build  # noqa: F401
