"""Plain-Python oracle of the host page allocator (test infrastructure only).

Restates the page-pool rules of AstrAI's cache layer (astrai/inference/cache.py:
PagePool, PrefixCache, TaskTable and PagedCache's task_* calls; design in
docs/guides/inference.md, "KVCache System") with Python sets, dicts and an
ordered dict as the LRU list, for comparison with the library's C++
allocator:

* allocation takes the lowest-numbered free page; with none free, the least
  recently used cached page is evicted (its content hash is forgotten);
* freeing the last reference keeps a page cached (in the LRU list) while its
  content hash is recorded, otherwise the page becomes free;
* a page's content hash is h <- (h * 31 + token) mod 2^64 over its tokens; a
  prompt lookup walks the full pages and stops at the first unknown hash.

Readings where the reference code is not self-consistent (the same in the
C++ allocator): a page referenced by a task is never in the LRU list (a
prefix hit leaves it; touching a page outside the list does nothing); a
hash recorded for a new page takes the entry from the page that held it,
which stops being a cached page; evicting a page forgets only the entry that
names that page.
"""
from collections import OrderedDict

MASK64 = (1 << 64) - 1


def page_hash(token_ids, page_idx, page_size):
    h = 0
    for t in token_ids[page_idx * page_size: page_idx * page_size + page_size]:
        h = (h * 31 + int(t)) & MASK64
    return h


class PoolOracle:
    def __init__(self, n_pages, page_size):
        self.n_pages = n_pages
        self.page_size = page_size
        self.free = set(range(n_pages))
        self.refs = [0] * n_pages
        self.lru = OrderedDict()          # cached pages, oldest first
        self.hash_of = {}                 # page -> hash
        self.page_of = {}                 # hash -> page
        self.tasks = {}                   # task id -> [pages, cached tokens]

    # -- pages -----------------------------------------------------------
    def _forget(self, p):
        h = self.hash_of.pop(p, None)
        if h is not None and self.page_of.get(h) == p:
            del self.page_of[h]

    def alloc(self):
        if self.free:
            p = min(self.free)
            self.free.remove(p)
        elif self.lru:
            p, _ = self.lru.popitem(last=False)
            self._forget(p)
        else:
            return -1
        self.refs[p] = 1
        return p

    def release(self, p):
        if not (0 <= p < self.n_pages) or self.refs[p] <= 0:
            return -1
        self.refs[p] -= 1
        if self.refs[p] == 0:
            if p in self.hash_of:
                self.lru[p] = None
            else:
                self.free.add(p)
        return 0

    def _take_ref(self, p):
        if self.refs[p] == 0:
            self.lru.pop(p, None)
        self.refs[p] += 1

    def _record(self, p, h):
        self._forget(p)
        q = self.page_of.get(h)
        if q is not None and q != p:
            del self.hash_of[q]
            if q in self.lru:
                del self.lru[q]
                self.free.add(q)
        self.page_of[h] = p
        self.hash_of[p] = h
        self.lru.pop(p, None)

    # -- tasks -----------------------------------------------------------
    def task_alloc(self, tid, prompt):
        if tid in self.tasks:
            return -1, 0
        ps = self.page_size
        hits = []
        for i in range(len(prompt) // ps):
            p = self.page_of.get(page_hash(prompt, i, ps))
            if p is None:
                break
            if p in self.lru:
                self.lru.move_to_end(p)
            hits.append(p)
        for p in hits:
            self._take_ref(p)
        cached = len(hits) * ps
        remaining = len(prompt) - cached
        pages = list(hits)
        for _ in range(-(-remaining // ps) if remaining > 0 else 0):
            p = self.alloc()
            if p < 0:
                for q in pages:
                    self.release(q)
                return -3, 0
            pages.append(p)
        self.tasks[tid] = [pages, cached]
        return 0, cached

    def task_free(self, tid):
        if tid not in self.tasks:
            return -1
        pages, _ = self.tasks.pop(tid)
        for p in pages:
            self.release(p)
        return 0

    def task_extend(self, tid, pos):
        if tid not in self.tasks or pos < 0:
            return -1
        pages = self.tasks[tid][0]
        while len(pages) < (pos + self.page_size) // self.page_size:
            p = self.alloc()
            if p < 0:
                return -3
            pages.append(p)
        return 0

    def task_record_hashes(self, tid, prompt, start=0):
        if tid not in self.tasks:
            return -1
        pages = self.tasks[tid][0]
        full = len(prompt) // self.page_size
        if full > len(pages):
            return -1
        for i in range(start, full):
            self._record(pages[i], page_hash(prompt, i, self.page_size))
        return 0

    def task_pages(self, tid):
        return list(self.tasks[tid][0]) if tid in self.tasks else None
