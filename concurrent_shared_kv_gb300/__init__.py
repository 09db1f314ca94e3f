"""GB300-native concurrent decode attention over a shared KV cache (Hogwild! Inference).

The compute lives in libhogwild.so (hand-written CUDA for sm_103a, C ABI in
include/hogwild.h); ``api`` is its ctypes binding and ``engine`` a thin
torch-facing wrapper that owns the workspace.
"""
from . import api  # noqa: F401
