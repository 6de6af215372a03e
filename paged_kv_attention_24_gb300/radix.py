"""ctypes binding of the host-side radix prefix cache (``include/msgl_radix.h``).

Argument marshalling only: the tree, the page states and the LRU eviction
live in ``csrc/radix_cache.cpp`` inside libmsgl_attn.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import ops

P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
SIGNATURES = {
    "msgl_radix_create": ([I32, I32], P),
    "msgl_radix_destroy": ([P], None),
    "msgl_radix_match": ([P, P, I32, P, I32, ctypes.POINTER(I64)], I32),
    "msgl_radix_alloc": ([P, I32, P], I32),
    "msgl_radix_insert": ([P, P, I32, P, I64], I32),
    "msgl_radix_release": ([P, I64, P, I32], I32),
    "msgl_radix_stats": ([P, ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(I32)], I32),
}
ERRORS = {-1: "bad argument", -2: "not enough free or evictable pages", -3: "unknown lease",
          -4: "page id outside the pool"}

_bound = False


def _lib():
    global _bound
    lib = ops.load()
    if not _bound:
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _bound = True
    return lib


class RadixError(RuntimeError):
    pass


def _arr(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise RadixError(f"{what}: {ERRORS.get(rc, rc)}")
    return rc


class RadixCache:
    """Radix tree of cached pages over a pool of ``num_pages`` pages of ``page_size`` tokens."""

    def __init__(self, page_size: int, num_pages: int):
        self.page_size, self.num_pages = int(page_size), int(num_pages)
        self._h = _lib().msgl_radix_create(self.page_size, self.num_pages)
        if not self._h:
            raise RadixError("bad cache arguments")

    def close(self):
        if self._h:
            _lib().msgl_radix_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens: Sequence[int]):
        """(matched token count, page ids of the match, lease)."""
        t = _arr(tokens)
        cap = len(t) // self.page_size
        out = np.zeros(max(cap, 1), dtype=np.int32)
        lease = I64(0)
        n = _check(_lib().msgl_radix_match(self._h, t.ctypes.data, len(t), out.ctypes.data, cap,
                                           ctypes.byref(lease)), "match")
        return n, out[: n // self.page_size].copy(), lease.value

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(int(n), 1), dtype=np.int32)
        _check(_lib().msgl_radix_alloc(self._h, int(n), out.ctypes.data), "alloc")
        return out[: int(n)].copy()

    def insert(self, tokens: Sequence[int], pages: Sequence[int], lease: int) -> int:
        t, p = _arr(tokens), _arr(pages)
        return _check(_lib().msgl_radix_insert(self._h, t.ctypes.data, len(t), p.ctypes.data, int(lease)),
                      "insert")

    def release(self, lease: int, pages: Sequence[int]) -> None:
        p = _arr(pages)
        _check(_lib().msgl_radix_release(self._h, int(lease), p.ctypes.data, len(p)), "release")

    def stats(self):
        f, c, pn = I32(0), I32(0), I32(0)
        _check(_lib().msgl_radix_stats(self._h, ctypes.byref(f), ctypes.byref(c), ctypes.byref(pn)), "stats")
        return {"free": f.value, "cached": c.value, "pinned": pn.value}

    def admit(self, tokens: Sequence[int]):
        """Match a new request's prefix and allocate pages for the rest.

        Returns (prefix_len, page ids covering all tokens, lease).
        """
        n, pre_pages, lease = self.match(tokens)
        need = -(-len(tokens) // self.page_size) - len(pre_pages)
        try:
            own = self.alloc(need)
        except RadixError:
            self.release(lease, [])
            raise
        return n, np.concatenate([pre_pages, own]).astype(np.int32), lease
