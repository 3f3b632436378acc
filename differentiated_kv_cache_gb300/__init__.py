"""Differentiated KV compaction (DiffKV) for one NVIDIA GB300 (sm_103a).

The product is libdkv.so (C ABI in include/dkv.h); ``dkv`` is its ctypes
binding, ``build`` compiles it in-tree with nvcc.
"""
from . import build
from .dkv import *  # noqa: F401,F403
