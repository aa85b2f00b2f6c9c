"""Collectives among N virtual ranks on one GB300: a CUDA library (libvcomm.so, C ABI in
include/vcomm.h) and its thin ctypes binding.

``vcomm`` holds the binding (vcommInit, vAllReduce, ... with the C names); ``build``
compiles the library in-tree for sm_103a; ``inputs`` draws the seeded synthetic buffers.
Importing the package loads nothing; the library is loaded on the first call.
"""
from . import build  # noqa: F401
