"""GB300-native MoE dispatch + combine on one GPU.

The compute path is the CUDA library libmoe.so (C ABI in include/moe.h,
kernels in csrc/); ``moe`` is its thin ctypes binding and ``inputs`` the
seeded synthetic workloads.  Importing the package does not load the CUDA
library; the first call into ``moe`` does, and raises if it is not built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "moe"]
