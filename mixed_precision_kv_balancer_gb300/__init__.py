"""MiKV mixed-precision KV cache hot path for GB300 (sm_103a).

The compute path is libmikv.so (hand-written CUDA, C ABI declared in
include/mikv.h); ``_lib`` binds its calls under their C names and ``cache``
sequences them per layer.  Importing this package does not load the library;
the first call does, and raises if it has not been built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "load"]


def load():
    """Load libmikv.so and return the binding module."""
    from . import _lib
    _lib.load()
    return _lib
