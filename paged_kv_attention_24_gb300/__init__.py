"""GB300-native paged-KV grouped-query attention (``libmsgl_attn``).

The compute lives in CUDA kernels for sm_103a behind a C ABI
(``include/msgl_attn.h``); :mod:`.ops` is a thin ctypes binding over it.
Importing the package does not load the library; the first call into
:mod:`.ops` does, and fails loudly if it has not been built.
"""
from __future__ import annotations

__all__ = ["ops", "workloads", "accounting"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
