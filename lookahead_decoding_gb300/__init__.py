"""Lookahead decoding on one GB300: the packed per-step target call behind a C ABI.

The compute lives in liblookahead.so (hand-written sm_103a CUDA); this package
holds its sources (csrc/), the in-tree build (build.py) and a ctypes binding
(_lib.py) whose functions carry the C entry points' names.
"""
from .build import build  # noqa: F401


def lib():
    """Import the binding (loads liblookahead.so; raises if it was not built)."""
    from . import _lib
    return _lib
