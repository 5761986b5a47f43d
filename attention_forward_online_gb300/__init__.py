"""libosattn for GB300: fused attention forward with online softmax, its
backward pass and the standalone row softmax.

The compute lives in hand-written CUDA kernels (csrc/) behind the C ABI in
include/osattn.h; ``osattn`` is the ctypes binding.  Importing this package
loads nothing; libosattn.so is loaded on first use and its absence is an
error, never a fallback.
"""
from . import inputs, osattn  # noqa: F401

__all__ = ["inputs", "osattn"]
