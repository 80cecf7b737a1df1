"""Python binding of the host page allocator (include/pkv_pool.h)."""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence

import numpy as np

from . import _lib


def _ids(tokens: Sequence[int]) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class PagePool:
    """Bitmask page allocator with reference counts, LRU eviction of cached
    pages and hash-based prefix reuse (C++; host only)."""

    def __init__(self, n_pages: int, page_size: int):
        self._lib = _lib.load()
        self._h = self._lib.pkv_pool_create(n_pages, page_size)
        if not self._h:
            raise ValueError("bad pool sizes")
        self.n_pages, self.page_size = n_pages, page_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pkv_pool_destroy(h)
            self._h = None

    def alloc(self) -> int:
        return self._lib.pkv_pool_page_alloc(self._h)

    def free(self, page: int) -> int:
        return self._lib.pkv_pool_page_free(self._h, page)

    @property
    def num_free(self) -> int:
        return self._lib.pkv_pool_num_free(self._h)

    @property
    def num_cached(self) -> int:
        return self._lib.pkv_pool_num_cached(self._h)

    def refcount(self, page: int) -> int:
        return self._lib.pkv_pool_refcount(self._h, page)

    def task_alloc(self, task_id: int, prompt: Sequence[int]):
        ids = _ids(prompt)
        cached = ctypes.c_int32(0)
        rc = self._lib.pkv_pool_task_alloc(self._h, task_id, _p(ids), ids.size, ctypes.byref(cached))
        return rc, cached.value

    def task_free(self, task_id: int) -> int:
        return self._lib.pkv_pool_task_free(self._h, task_id)

    def task_extend(self, task_id: int, pos: int) -> int:
        return self._lib.pkv_pool_task_extend(self._h, task_id, pos)

    def task_record_hashes(self, task_id: int, prompt: Sequence[int], start_logical_page: int = 0) -> int:
        ids = _ids(prompt)
        return self._lib.pkv_pool_task_record_hashes(self._h, task_id, _p(ids), ids.size,
                                                     start_logical_page)

    def task_pages(self, task_id: int) -> Optional[List[int]]:
        n = self._lib.pkv_pool_task_pages(self._h, task_id, None, 0)
        if n < 0:
            return None
        out = np.zeros(max(n, 1), np.int32)
        self._lib.pkv_pool_task_pages(self._h, task_id, _p(out), n)
        return out[:n].tolist()

    def task_slots(self, task_id: int, n_tokens: int) -> np.ndarray:
        out = np.zeros(max(n_tokens, 1), np.int32)
        _lib.check(self._lib.pkv_pool_task_slots(self._h, task_id, n_tokens, _p(out)), "pkv_pool_task_slots")
        return out[:n_tokens]


def page_hash(tokens: Sequence[int], page_idx: int, page_size: int) -> int:
    ids = _ids(tokens)
    return _lib.load().pkv_pool_page_hash(_p(ids), ids.size, page_idx, page_size)
