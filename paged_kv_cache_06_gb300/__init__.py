"""GB300-native paged KV-cache decode attention.

The compute path is a C-ABI shared library of hand-written CUDA kernels for
sm_103a (``libpagedkv.so``, built from ``csrc/``); ``ops`` is a thin ctypes
binding over it (argument marshalling only).  PyTorch supplies device memory
and streams.  The library is loaded on first use, and every op raises if it
is missing: there is no CPU fallback.
"""
from __future__ import annotations

__all__ = ["ops", "workloads", "block_manager"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
