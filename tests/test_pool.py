"""Host page allocator: the Python oracle pinned by hand-worked scenarios and a
closed form, then the C++ allocator compared with it operation by operation.

Rules (AstrAI astrai/inference/cache.py: PagePool, PrefixCache, TaskTable and
PagedCache.task_*; docs/guides/inference.md, "KVCache System"): lowest free
page first; last reference freed -> page kept in an LRU list while its content
hash is recorded, else freed; out of free pages -> evict the least recently
used cached page; prefix lookup walks full pages until the first miss.
"""
import numpy as np
import pytest

from oracle.pool_oracle import MASK64, PoolOracle, page_hash
from paged_kv_cache_loc_gb300 import build
from paged_kv_cache_loc_gb300 import pool as P


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()


# ---------------------------------------------------------------------------
# pins of the oracle
# ---------------------------------------------------------------------------

def test_page_hash_closed_form():
    """h = sum_i t_i 31^(n-1-i) mod 2^64 over the page's tokens (Horner's rule)."""
    rng = np.random.Generator(np.random.PCG64(1))
    toks = rng.integers(0, 2**31 - 1, 50).tolist()
    for ps in (1, 4, 16):
        for i in range(0, 50 // ps + 1):
            seg = toks[i * ps: i * ps + ps]
            closed = sum(t * pow(31, len(seg) - 1 - k, 1 << 64) for k, t in enumerate(seg)) % (1 << 64)
            assert page_hash(toks, i, ps) == closed
            assert P.page_hash(toks, i, ps) == closed   # the C++ hash too
    assert page_hash([-1], 0, 1) == MASK64              # negative ids wrap like uint64


def test_oracle_lowest_first_and_lru_eviction():
    o = PoolOracle(4, 2)
    assert [o.alloc() for _ in range(4)] == [0, 1, 2, 3]
    assert o.alloc() == -1
    o.release(2)
    assert o.alloc() == 2                               # freed page comes back
    # make pages 1 and 3 cached copies of prompts, then release them
    o.tasks["a"] = [[1], 0]
    o.tasks["b"] = [[3], 0]
    o.task_record_hashes("a", [7, 8])
    o.task_record_hashes("b", [9, 9])
    o.release(1)
    o.release(3)
    assert list(o.lru) == [1, 3]                        # cached, oldest first
    o.release(0)
    assert o.alloc() == 0                               # free page before eviction
    assert o.alloc() == 1                               # then the oldest cached page
    assert page_hash([7, 8], 0, 2) not in o.page_of     # its content was forgotten
    assert o.alloc() == 3 and o.alloc() == -1


def test_oracle_prefix_reuse_and_rollback():
    o = PoolOracle(6, 4)
    prompt = list(range(10))                            # 2 full pages + 2 tokens
    assert o.task_alloc(1, prompt) == (0, 0)
    assert o.task_pages(1) == [0, 1, 2]
    o.task_record_hashes(1, prompt)
    rc, cached = o.task_alloc(2, prompt[:8] + [99, 98, 97])   # shares 2 full pages
    assert (rc, cached) == (0, 8) and o.task_pages(2)[:2] == [0, 1]
    assert o.refs[0] == 2 and o.refs[1] == 2
    # not enough pages: every reference taken is returned
    before = (set(o.free), list(o.refs), list(o.lru))
    assert o.task_alloc(3, prompt[:8] + list(range(100, 120))) == (-3, 0)
    assert (set(o.free), list(o.refs), list(o.lru)) == before
    o.task_free(1)
    o.task_free(2)
    assert sorted(o.lru) == [0, 1] and 2 in o.free       # hashed pages stay cached
    assert o.task_alloc(4, prompt) == (0, 8)             # found again after both ended
    assert 0 not in o.lru and 1 not in o.lru             # in use: not evictable


def test_oracle_extend():
    o = PoolOracle(4, 4)
    o.task_alloc(1, [1, 2, 3])
    assert o.task_extend(1, 3) == 0 and len(o.task_pages(1)) == 1
    assert o.task_extend(1, 4) == 0 and len(o.task_pages(1)) == 2
    assert o.task_extend(1, 15) == 0 and len(o.task_pages(1)) == 4
    assert o.task_extend(1, 16) == -3


# ---------------------------------------------------------------------------
# C++ allocator == oracle
# ---------------------------------------------------------------------------

def _state(pool_c, pool_o, tids):
    assert pool_c.num_free == len(pool_o.free)
    assert pool_c.num_cached == len(pool_o.lru)
    for p in range(pool_o.n_pages):
        assert pool_c.refcount(p) == pool_o.refs[p]
    for t in tids:
        assert pool_c.task_pages(t) == pool_o.task_pages(t)


@pytest.mark.parametrize("seed,n_pages,page_size", [(0, 64, 4), (1, 37, 16), (2, 200, 1), (3, 16, 8)])
def test_cpp_pool_matches_oracle_on_random_churn(seed, n_pages, page_size):
    rng = np.random.Generator(np.random.PCG64(seed))
    c, o = P.PagePool(n_pages, page_size), PoolOracle(n_pages, page_size)
    prefixes = [rng.integers(0, 50, rng.integers(0, 40)).tolist() for _ in range(5)]
    live, prompts, next_id = [], {}, 0
    for step in range(600):
        op = rng.integers(0, 5)
        if op <= 1:   # new task with a prompt sharing one of a few prefixes
            prompt = prefixes[rng.integers(0, 5)] + rng.integers(0, 50, rng.integers(0, 30)).tolist()
            rc_c = c.task_alloc(next_id, prompt)
            rc_o = o.task_alloc(next_id, prompt)
            assert rc_c == rc_o, (step, rc_c, rc_o)
            if rc_o[0] == 0:
                live.append(next_id)
                prompts[next_id] = prompt
            next_id += 1
        elif op == 2 and live:   # prefill done: record hashes
            t = live[rng.integers(0, len(live))]
            assert c.task_record_hashes(t, prompts[t]) == o.task_record_hashes(t, prompts[t])
        elif op == 3 and live:   # decode growth
            t = live[rng.integers(0, len(live))]
            pos = len(prompts[t]) + int(rng.integers(0, 3 * page_size))
            assert c.task_extend(t, pos) == o.task_extend(t, pos)
        elif live:              # task finished
            t = live.pop(rng.integers(0, len(live)))
            assert c.task_free(t) == o.task_free(t) == 0
        _state(c, o, live)
    for t in live:
        n = len(o.task_pages(t)) * page_size
        slots = c.task_slots(t, n)
        pages = o.task_pages(t)
        assert slots.tolist() == [pages[j // page_size] * page_size + j % page_size for j in range(n)]


def test_cpp_pool_argument_errors():
    c = P.PagePool(4, 4)
    assert c.free(0) < 0                     # no reference held
    assert c.task_free(9) < 0
    assert c.task_extend(9, 0) < 0
    assert c.task_alloc(1, [1, 2])[0] == 0
    assert c.task_alloc(1, [1, 2])[0] < 0   # duplicate task id
    assert c.task_record_hashes(1, list(range(40))) < 0   # more full pages than the task has
    with pytest.raises(Exception):
        c.task_slots(1, 5)                   # one page covers 4 slots only
