/*
 * pkv_pool.h -- host-side page allocator for the paged KV pool.
 *
 * Follows AstrAI's cache layer (astrai/inference/cache.py: PagePool,
 * PrefixCache, TaskTable and the PagedCache facade's task_* calls; design in
 * docs/guides/inference.md, "KVCache System": "bitmask-based page allocator +
 * ref-count + LRU" and "hash-based prefix matching"):
 *   - pages are handed out lowest-index-first from a free bitmask;
 *   - each page has a reference count; a page whose count drops to zero is
 *     kept in an LRU list while its contents are reachable through the
 *     prefix cache (so a later prompt with the same prefix reuses it), and is
 *     returned to the bitmask otherwise;
 *   - when the bitmask is empty, the least recently used cached page is
 *     evicted (its prefix-cache entry is forgotten) and handed out;
 *   - a page's content hash is h = (h*31 + token) mod 2^64 over its tokens;
 *     a prompt's prefix lookup walks its full pages and stops at the first
 *     page whose hash is unknown.
 * Two readings where the reference code is not self-consistent:
 *   - a page that a task references is never in the LRU list (a prefix hit
 *     leaves it), so eviction never takes a page in use;
 *   - recording a hash that already names another page moves the entry to the
 *     new page and the other page stops being a cached page; evicting a page
 *     forgets only the entry that names that page.
 *
 * Host only: no CUDA call, thread-compatible (one pool per thread or external
 * locking).  Return codes are those of pkv.h (PKV_OK, PKV_ERR_ARG,
 * PKV_ERR_WORKSPACE for "no page available").
 */
#ifndef PKV_POOL_H_
#define PKV_POOL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_pool pkv_pool;

/* A pool of n_pages pages of page_size token slots (page p owns slots
 * [p*page_size, (p+1)*page_size)).  NULL on bad sizes or allocation failure. */
pkv_pool *pkv_pool_create(int32_t n_pages, int32_t page_size);
void pkv_pool_destroy(pkv_pool *pool);

/* One page with reference count 1: the lowest free page, else the least
 * recently used cached page (evicted), else -1. */
int32_t pkv_pool_page_alloc(pkv_pool *pool);

/* Drop one reference to `page` (PKV_ERR_ARG if it has none). */
int pkv_pool_page_free(pkv_pool *pool, int32_t page);

/* Counters: pages in the free bitmask; cached pages (refcount 0, in the LRU). */
int32_t pkv_pool_num_free(const pkv_pool *pool);
int32_t pkv_pool_num_cached(const pkv_pool *pool);
int32_t pkv_pool_refcount(const pkv_pool *pool, int32_t page);

/* Content hash of logical page `page_idx` of a token sequence. */
uint64_t pkv_pool_page_hash(const int32_t *token_ids, int32_t n_tokens, int32_t page_idx,
                            int32_t page_size);

/*
 * Give task `task_id` pages for its prompt: full pages found in the prefix
 * cache are shared (reference +1), the rest are allocated.  *cached_tokens
 * receives the number of prompt tokens already in the cache.  On failure
 * every reference taken is dropped again and PKV_ERR_WORKSPACE is returned;
 * PKV_ERR_ARG if the task exists.
 */
int pkv_pool_task_alloc(pkv_pool *pool, int64_t task_id, const int32_t *prompt_ids,
                        int32_t n_tokens, int32_t *cached_tokens);

/* Release every page of the task and forget it (PKV_ERR_ARG if unknown). */
int pkv_pool_task_free(pkv_pool *pool, int64_t task_id);

/* Grow the task's page list to cover position `pos` (decode).  Pages added
 * before a failure stay with the task.  PKV_ERR_WORKSPACE when out of pages. */
int pkv_pool_task_extend(pkv_pool *pool, int64_t task_id, int32_t pos);

/* Record the content hashes of the task's full prompt pages from
 * `start_logical_page` on, making them findable by later prefix lookups. */
int pkv_pool_task_record_hashes(pkv_pool *pool, int64_t task_id, const int32_t *prompt_ids,
                                int32_t n_tokens, int32_t start_logical_page);

/* The task's page list (up to max_pages entries written); returns its length,
 * or -1 if the task is unknown. */
int32_t pkv_pool_task_pages(const pkv_pool *pool, int64_t task_id, int32_t *pages_out,
                            int32_t max_pages);

/* The task's req_to_token row: slots_out[j] = page[j / page_size] * page_size +
 * j % page_size for j < n_tokens (PKV_ERR_ARG if the pages do not cover it). */
int pkv_pool_task_slots(const pkv_pool *pool, int64_t task_id, int32_t n_tokens,
                        int32_t *slots_out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_POOL_H_ */
