"""Query-aware sparse KV-block selection and sparse decode attention on GB300.

The compute path is libkvsel.so (hand-written CUDA for sm_103a, C ABI in
include/kvsel.h); ``kvsel`` is its ctypes binding and ``runtime`` holds the
device buffers around it. The library is loaded on first use and its absence
is an error: there is no CPU path.
"""
from . import kvsel  # noqa: F401
from .kvsel import KvselError  # noqa: F401

__all__ = ["kvsel", "KvselError"]
