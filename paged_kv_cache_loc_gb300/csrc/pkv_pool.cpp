// pkv_pool.cpp -- host-side page allocator (see include/pkv_pool.h).
//
// Free pages: a bitmask of 64-bit words searched from a low-water hint, so
// the lowest free page comes out first.  Cached pages (reference count 0,
// content still findable): an intrusive doubly linked LRU list over page
// indices, oldest at the head.  Prefix cache: page -> hash and hash -> page
// maps kept as a bijection.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "pkv_pool.h"

namespace {

struct Task {
    std::vector<int32_t> pages;
    int32_t cached = 0;
};

}  // namespace

struct pkv_pool {
    int32_t n_pages = 0;
    int32_t page_size = 0;
    std::vector<uint64_t> free_bits;   // bit p set: page p is free
    int32_t free_hint = 0;             // no free bit below word free_hint
    int32_t n_free = 0;
    std::vector<int32_t> refs;
    // LRU of cached pages: prev/next links, -1 terminated; in_lru marks members
    std::vector<int32_t> prev, next;
    std::vector<uint8_t> in_lru;
    int32_t lru_head = -1, lru_tail = -1, n_cached = 0;
    // prefix cache
    std::vector<uint8_t> has_hash;
    std::vector<uint64_t> hash_of;
    std::unordered_map<uint64_t, int32_t> page_of_hash;
    std::unordered_map<int64_t, Task> tasks;

    bool valid(int32_t p) const { return p >= 0 && p < n_pages; }

    void set_free(int32_t p) {
        free_bits[p >> 6] |= 1ull << (p & 63);
        if ((p >> 6) < free_hint) free_hint = p >> 6;
        ++n_free;
    }
    int32_t take_lowest_free() {
        const int32_t words = static_cast<int32_t>(free_bits.size());
        for (int32_t w = free_hint; w < words; ++w) {
            if (free_bits[w]) {
                const int b = __builtin_ctzll(free_bits[w]);
                free_bits[w] &= free_bits[w] - 1;
                free_hint = w;
                --n_free;
                return w * 64 + b;
            }
        }
        free_hint = words;
        return -1;
    }

    void lru_push_back(int32_t p) {
        prev[p] = lru_tail;
        next[p] = -1;
        if (lru_tail >= 0) next[lru_tail] = p; else lru_head = p;
        lru_tail = p;
        in_lru[p] = 1;
        ++n_cached;
    }
    void lru_remove(int32_t p) {
        if (!in_lru[p]) return;
        if (prev[p] >= 0) next[prev[p]] = next[p]; else lru_head = next[p];
        if (next[p] >= 0) prev[next[p]] = prev[p]; else lru_tail = prev[p];
        prev[p] = next[p] = -1;
        in_lru[p] = 0;
        --n_cached;
    }
    void lru_touch(int32_t p) {
        if (!in_lru[p]) return;
        lru_remove(p);
        lru_push_back(p);
    }

    // the page's contents are no longer findable
    void forget_hash(int32_t p) {
        if (!has_hash[p]) return;
        auto it = page_of_hash.find(hash_of[p]);
        if (it != page_of_hash.end() && it->second == p) page_of_hash.erase(it);
        has_hash[p] = 0;
    }

    int32_t alloc() {
        int32_t p = take_lowest_free();
        if (p < 0) {
            if (lru_head < 0) return -1;
            p = lru_head;   // evict the least recently used cached page
            lru_remove(p);
            forget_hash(p);
        }
        refs[p] = 1;
        return p;
    }

    // drop one reference; an unreferenced page stays cached if findable
    int release(int32_t p) {
        if (!valid(p) || refs[p] <= 0) return PKV_ERR_ARG;
        if (--refs[p] == 0) {
            if (has_hash[p]) lru_push_back(p);
            else set_free(p);
        }
        return PKV_OK;
    }

    void take_ref(int32_t p) {
        if (refs[p] == 0) lru_remove(p);   // a referenced page is never evictable
        ++refs[p];
    }

    void record(int32_t p, uint64_t h) {
        forget_hash(p);
        auto it = page_of_hash.find(h);
        if (it != page_of_hash.end() && it->second != p) {
            // the other page stops being a cached copy of this content
            const int32_t q = it->second;
            has_hash[q] = 0;
            if (in_lru[q]) {
                lru_remove(q);
                set_free(q);
            }
        }
        page_of_hash[h] = p;
        hash_of[p] = h;
        has_hash[p] = 1;
        lru_remove(p);
    }
};

extern "C" {

uint64_t pkv_pool_page_hash(const int32_t *token_ids, int32_t n_tokens, int32_t page_idx,
                            int32_t page_size) {
    uint64_t h = 0;
    if (!token_ids || page_size <= 0 || page_idx < 0) return h;
    const int64_t start = static_cast<int64_t>(page_idx) * page_size;
    const int64_t end = start + page_size < n_tokens ? start + page_size : n_tokens;
    for (int64_t i = start; i < end; ++i)
        h = h * 31u + static_cast<uint64_t>(static_cast<int64_t>(token_ids[i]));
    return h;
}

pkv_pool *pkv_pool_create(int32_t n_pages, int32_t page_size) {
    if (n_pages <= 0 || page_size <= 0) return nullptr;
    if (static_cast<int64_t>(n_pages) * page_size > INT32_MAX) return nullptr;   // slots are int32
    pkv_pool *pool = new (std::nothrow) pkv_pool();
    if (!pool) return nullptr;
    try {
        pool->n_pages = n_pages;
        pool->page_size = page_size;
        pool->free_bits.assign((n_pages + 63) / 64, 0);
        for (int32_t p = 0; p < n_pages; ++p) pool->set_free(p);
        pool->free_hint = 0;
        pool->refs.assign(n_pages, 0);
        pool->prev.assign(n_pages, -1);
        pool->next.assign(n_pages, -1);
        pool->in_lru.assign(n_pages, 0);
        pool->has_hash.assign(n_pages, 0);
        pool->hash_of.assign(n_pages, 0);
    } catch (...) {
        delete pool;
        return nullptr;
    }
    return pool;
}

void pkv_pool_destroy(pkv_pool *pool) { delete pool; }

int32_t pkv_pool_page_alloc(pkv_pool *pool) { return pool ? pool->alloc() : -1; }

int pkv_pool_page_free(pkv_pool *pool, int32_t page) {
    return pool ? pool->release(page) : PKV_ERR_ARG;
}

int32_t pkv_pool_num_free(const pkv_pool *pool) { return pool ? pool->n_free : 0; }
int32_t pkv_pool_num_cached(const pkv_pool *pool) { return pool ? pool->n_cached : 0; }
int32_t pkv_pool_refcount(const pkv_pool *pool, int32_t page) {
    return pool && pool->valid(page) ? pool->refs[page] : -1;
}

int pkv_pool_task_alloc(pkv_pool *pool, int64_t task_id, const int32_t *prompt_ids,
                        int32_t n_tokens, int32_t *cached_tokens) {
    if (!pool || n_tokens < 0 || (n_tokens > 0 && !prompt_ids)) return PKV_ERR_ARG;
    if (pool->tasks.count(task_id)) return PKV_ERR_ARG;
    const int32_t ps = pool->page_size;
    Task t;
    // prefix lookup over full pages, stopping at the first unknown page
    const int32_t full = n_tokens / ps;
    for (int32_t i = 0; i < full; ++i) {
        auto it = pool->page_of_hash.find(pkv_pool_page_hash(prompt_ids, n_tokens, i, ps));
        if (it == pool->page_of_hash.end()) break;
        pool->lru_touch(it->second);
        t.pages.push_back(it->second);
    }
    for (int32_t p : t.pages) pool->take_ref(p);
    t.cached = static_cast<int32_t>(t.pages.size()) * ps;
    const int32_t remaining = n_tokens - t.cached;
    const int32_t n_new = remaining > 0 ? (remaining + ps - 1) / ps : 0;
    for (int32_t i = 0; i < n_new; ++i) {
        const int32_t p = pool->alloc();
        if (p < 0) {
            for (int32_t q : t.pages) pool->release(q);   // roll back
            return PKV_ERR_WORKSPACE;
        }
        t.pages.push_back(p);
    }
    if (cached_tokens) *cached_tokens = t.cached;
    pool->tasks.emplace(task_id, std::move(t));
    return PKV_OK;
}

int pkv_pool_task_free(pkv_pool *pool, int64_t task_id) {
    if (!pool) return PKV_ERR_ARG;
    auto it = pool->tasks.find(task_id);
    if (it == pool->tasks.end()) return PKV_ERR_ARG;
    for (int32_t p : it->second.pages) pool->release(p);
    pool->tasks.erase(it);
    return PKV_OK;
}

int pkv_pool_task_extend(pkv_pool *pool, int64_t task_id, int32_t pos) {
    if (!pool || pos < 0) return PKV_ERR_ARG;
    auto it = pool->tasks.find(task_id);
    if (it == pool->tasks.end()) return PKV_ERR_ARG;
    const int64_t needed = (static_cast<int64_t>(pos) + pool->page_size) / pool->page_size;
    std::vector<int32_t> &pages = it->second.pages;
    while (static_cast<int64_t>(pages.size()) < needed) {
        const int32_t p = pool->alloc();
        if (p < 0) return PKV_ERR_WORKSPACE;
        pages.push_back(p);
    }
    return PKV_OK;
}

int pkv_pool_task_record_hashes(pkv_pool *pool, int64_t task_id, const int32_t *prompt_ids,
                                int32_t n_tokens, int32_t start_logical_page) {
    if (!pool || n_tokens < 0 || (n_tokens > 0 && !prompt_ids) || start_logical_page < 0)
        return PKV_ERR_ARG;
    auto it = pool->tasks.find(task_id);
    if (it == pool->tasks.end()) return PKV_ERR_ARG;
    const std::vector<int32_t> &pages = it->second.pages;
    const int32_t full = n_tokens / pool->page_size;
    if (full > static_cast<int32_t>(pages.size())) return PKV_ERR_ARG;
    for (int32_t i = start_logical_page; i < full; ++i)
        pool->record(pages[i], pkv_pool_page_hash(prompt_ids, n_tokens, i, pool->page_size));
    return PKV_OK;
}

int32_t pkv_pool_task_pages(const pkv_pool *pool, int64_t task_id, int32_t *pages_out,
                            int32_t max_pages) {
    if (!pool) return -1;
    auto it = pool->tasks.find(task_id);
    if (it == pool->tasks.end()) return -1;
    const std::vector<int32_t> &pages = it->second.pages;
    for (int32_t i = 0; i < max_pages && i < static_cast<int32_t>(pages.size()); ++i) pages_out[i] = pages[i];
    return static_cast<int32_t>(pages.size());
}

int pkv_pool_task_slots(const pkv_pool *pool, int64_t task_id, int32_t n_tokens,
                        int32_t *slots_out) {
    if (!pool || n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PKV_ERR_ARG;
    auto it = pool->tasks.find(task_id);
    if (it == pool->tasks.end()) return PKV_ERR_ARG;
    const std::vector<int32_t> &pages = it->second.pages;
    const int32_t ps = pool->page_size;
    if (static_cast<int64_t>(pages.size()) * ps < n_tokens) return PKV_ERR_ARG;
    for (int32_t j = 0; j < n_tokens; ++j) slots_out[j] = pages[j / ps] * ps + j % ps;
    return PKV_OK;
}

}  // extern "C"
