/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache hot path.
 *
 * The operations and names come from AstrAI's inference design
 * (docs/guides/inference.md):
 *   - "KV Cache": decode attention o_n = sum_j softmax(q_n k_j / sqrt(d_k)) v_j;
 *     RoPE is applied before the cache write;
 *   - "KVCache System": KVStorage k_buffer / v_buffer [n_layers, size,
 *     n_kv_heads, head_dim]; ReqToTokenPool req_to_token [num_reqs,
 *     max_ctx_len] (logical position -> physical token slot); the KVCache
 *     dataclass fields req_pool_indices, seq_lens, out_cache_loc, max_len,
 *     kv_indptr, qo_indptr; the write k_buffer[layer_id, out_cache_loc] = k;
 *   - "Attention Backend": decode writes K/V then attends through req_to_token
 *     with page_size 1; prefill writes K/V then attends over a ragged batch
 *     addressed by qo_indptr / kv_indptr;
 *   - "Rotary Embedding Backend": freqs_cis [max_len, dim/2, 2] f32 (cos, sin).
 * The commit log under tests/inference/test_cache.py fixes int32 page-table,
 * request-row and cache-location indices, and a workspace allocated once that
 * owns the split-K partials decode_o_part / decode_ml_part so that CUDA-graph
 * replay sees stable addresses.
 *
 * Conventions for every entry point:
 *   - All tensors are caller-owned, row-major and contiguous, in memory the
 *     GPU can address: device or managed memory, or registered (pinned)
 *     host memory mapped at the same address.  The pool, the index tables
 *     and the workspace belong in device memory; a step's small inputs and
 *     outputs (q, o, the new K/V rows, seq_lens, kv_indptr, qo_indptr,
 *     req_pool_indices, out_cache_loc) may stay in pinned host memory, which
 *     the kernels then read and write in place over the host link (on a
 *     Grace-Blackwell node: NVLink-C2C).  Any other address (unregistered
 *     host memory, say) returns PKV_ERR_ARG before anything is enqueued.
 *     The library never allocates, frees or copies host<->device.
 *   - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Work is enqueued asynchronously; the call returns once enqueued.
 *   - Return value: PKV_OK or a negative PKV_ERR_* code.  Errors the host can
 *     see (null pointers, shapes, sizes, alignment, unsupported variants) are
 *     returned before anything is enqueued.  Errors in device-resident data
 *     (a slot outside [0, size), a request row outside [0, num_reqs), a length
 *     beyond max_ctx_len / max_len, kv_len < q_len) never fault: the kernel
 *     substitutes a safe index, records the first such error in a per-device
 *     error word and finishes; pkv_last_device_error() reports it.  Results
 *     of a call that recorded such an error are unspecified.
 *   - Nothing traps, aborts or waits without a bound.
 *   - The library looks up the device addresses of its own device-resident
 *     objects (the error word, the array of pkv_paged_decode_noalloc) once
 *     per device and keeps them for the life of the process.  After
 *     cudaDeviceReset() on a device those addresses are stale: make no
 *     further pkv_* call on that device in the same process.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage element type of k_buffer / v_buffer; q, k, v and o use the same. */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

enum {
    PKV_OK = 0,
    PKV_ERR_ARG = -1,         /* bad pointer, shape, size, alignment or index range */
    PKV_ERR_UNSUPPORTED = -2, /* valid request that this build has no kernel for */
    PKV_ERR_WORKSPACE = -3,   /* workspace missing, uninitialised or too small */
    PKV_ERR_INDEX = -4,       /* device data out of range (from pkv_last_device_error) */
    PKV_ERR_CUDA = -5         /* a CUDA runtime call or launch failed */
};

/*
 * The KVCache dataclass of "KVCache System", as plain pointers and sizes.
 *   k_buffer, v_buffer  [n_layers, size, n_kv_heads, head_dim] of dtype; the
 *                       row of (layer, slot) is n_kv_heads*head_dim elements.
 *   req_to_token        int32 [num_reqs, max_ctx_len]: physical slot of each
 *                       logical position of each request row.  page_size > 1
 *                       pools are expressed per token (a page is a run of
 *                       page_size consecutive slots).
 *   req_pool_indices    int32 [batch]: request row of each batch entry.
 *   seq_lens            int32 [batch]: decode context length of each entry,
 *                       INCLUDING the token written this step.
 *   kv_indptr           int32 [batch + 1]: prefix sums of the kv lengths
 *                       (kv_indptr[0] = 0); in prefill the kv length of entry b
 *                       is kv_indptr[b+1] - kv_indptr[b] (cached prefix + new
 *                       tokens).  In decode it is optional: when given, it
 *                       must equal the prefix sums of seq_lens, and the
 *                       automatic plan splits all tokens of the batch evenly
 *                       across the SMs (an entry whose differences disagree
 *                       with seq_lens is a device-data error).
 *   qo_indptr           int32 [batch + 1]: prefix sums of the query lengths
 *                       (prefill only; NULL in decode).
 *   out_cache_loc       int32 [n_new]: destination slot of each new token, in
 *                       qo_indptr order (the pages' [batch, seq_len] flattened).
 *   batch               number of batch entries.
 *   max_len             host-side upper bound of seq_lens (decode) or of the kv
 *                       lengths (prefill): the pages pass max(seq_lens) on the
 *                       host so that no device sync is needed.  Launch grids
 *                       are sized from it.
 */
typedef struct pkv_kvcache {
    void *k_buffer;
    void *v_buffer;
    int32_t dtype;            /* pkv_dtype */
    int32_t n_layers;
    int32_t n_kv_heads;
    int32_t head_dim;
    int64_t size;
    const int32_t *req_to_token;
    int32_t num_reqs;
    int32_t max_ctx_len;
    const int32_t *req_pool_indices;
    const int32_t *seq_lens;
    const int32_t *kv_indptr;
    const int32_t *qo_indptr;
    const int32_t *out_cache_loc;
    int32_t batch;
    int32_t max_len;
} pkv_kvcache;

/*
 * Caller-owned workspace for the decode split-K partials (the pages'
 * decode_o_part / decode_ml_part):
 *   o_part   float [max_batch, n_heads, max_splits, head_dim]: normalised
 *            attention output of each split of each (entry, head);
 *   ml_part  float [max_batch, n_heads, max_splits, 2]: (running max in base-2
 *            units of the scaled score, softmax denominator) of each split.
 * Allocate pkv_workspace_bytes(...) bytes of device memory once (256-byte
 * aligned, e.g. straight from cudaMalloc), describe it with
 * pkv_workspace_init(), and pass the same descriptor to every call so that
 * the device addresses stay fixed across CUDA-graph replays.  No call needs
 * its contents to persist between calls; calls that share a workspace must not
 * overlap on the GPU.
 */
typedef struct pkv_workspace {
    void *base;
    size_t bytes;
    int32_t max_batch;
    int32_t n_heads;
    int32_t head_dim;
    int32_t max_splits;
    float *o_part;
    float *ml_part;
    uint32_t magic;           /* set by pkv_workspace_init */
} pkv_workspace;

/* Bytes needed for a workspace of these dimensions (0 if any is < 1). */
size_t pkv_workspace_bytes(int32_t max_batch, int32_t n_heads, int32_t head_dim,
                           int32_t max_splits);

/* Fill *out to describe `base`.  PKV_ERR_ARG on null / misaligned base or bad
 * dimensions, PKV_ERR_WORKSPACE if `bytes` is smaller than required. */
int pkv_workspace_init(void *base, size_t bytes, int32_t max_batch, int32_t n_heads,
                       int32_t head_dim, int32_t max_splits, pkv_workspace *out);

/*
 * K/V cache write ("KVCache System": k_buffer[layer_id, out_cache_loc] = k):
 * for i in [0, n_new): row (layer_id, c->out_cache_loc[i]) of c->k_buffer
 * (resp. v_buffer) becomes k[i] (resp. v[i]).  k, v: [n_new, n_kv_heads,
 * head_dim] of c->dtype.  Bit-exact copy.  Requires 16-byte aligned buffers
 * and a row of n_kv_heads*head_dim elements that is a multiple of 16 bytes.
 * Duplicate destination slots give an unspecified one of the rows.  n_new = 0
 * is a no-op.  Reads c->out_cache_loc, c->size, c->n_layers, the buffers and
 * shape fields only.
 */
int pkv_kv_write(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                 int32_t n_new, void *stream);

/*
 * Fused rotary embedding + K/V cache write ("KV Cache": RoPE before the
 * write; "Rotary Embedding Backend": freqs_cis [max_pos, head_dim/2, 2] f32).
 * Row i of k is rotated pairwise, (k[2e] + i k[2e+1]) * (cos + i sin) with
 * (cos, sin) = freqs_cis[positions[i], e], rounded once to the storage dtype,
 * and written like pkv_kv_write; v is copied unchanged.  positions: int32
 * [n_new] device array (a position outside [0, max_pos) is a device-data
 * error).  head_dim must be even.
 */
int pkv_rope_kv_write(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                      int32_t n_new, const float *freqs_cis, int32_t max_pos,
                      const int32_t *positions, void *stream);

/*
 * Paged decode attention ("KV Cache" formula; "Attention Backend" decode path).
 * For each entry b < c->batch with request row r = c->req_pool_indices[b] and
 * context n = c->seq_lens[b], and each query head h < n_heads:
 *   o[b, h] = sum_{j<n} softmax_j(sm_scale * q[b,h] . K[slot_j, h/G]) V[slot_j, h/G],
 *   slot_j = c->req_to_token[r, j],  G = n_heads / c->n_kv_heads,
 * with K/V the rows of layer `layer_id`.  q, o: [batch, n_heads, head_dim] of
 * c->dtype; o must not alias q.  n = 0 gives o = 0.  Accumulation in fp32,
 * one rounding to the output dtype.  The work is split and the partials go
 * to the workspace, merged by a second kernel:
 *   - with c->kv_indptr (bf16, n_kv_heads in {1, 2, 4, 8}): the tokens of the
 *     whole batch, [0, kv_indptr[batch]), are divided evenly among up to one
 *     CTA per SM; the workspace must hold (CTAs + batch) x n_heads partial
 *     rows (else the chunked plan below is used);
 *   - otherwise each context is cut into chunks whose size is chosen on the
 *     host from c->max_len, c->batch and the SM count.
 * Without a workspace only single-split plans are possible.
 * Supported: head_dim 64 or 128, G in {1, 2, 4, 8}.
 */
int pkv_paged_decode(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                     int32_t n_heads, float sm_scale, const pkv_workspace *ws, void *stream);

/*
 * pkv_paged_decode with a shared prefix stated: the first shared_len
 * positions of every request row of the batch (req_to_token[r, 0 ..
 * shared_len), r = c->req_pool_indices[b]) hold the same slots, as when the
 * prefix cache ("KVCache System") hands several tasks the same pages.  Same
 * operation and result as pkv_paged_decode; with the balanced plan, 8 kv
 * heads, shared_len >= 64, batch >= 2 and room in the workspace the shared
 * rows are read once per launch at head_dim 128 and once per group of 16 / G
 * requests at head_dim 64 (see pkv_paged_decode_pages for how, and for the
 * workspace it needs), otherwise the statement is ignored.  Every seq_len
 * must be >= shared_len; a shorter context, or a row whose leading slots
 * differ from the first entry's (head_dim 128) or its group's (head_dim
 * 64), is a device-data error.  shared_len < 0, or shared_len > c->max_len,
 * returns PKV_ERR_ARG.
 */
int pkv_paged_decode_shared(const pkv_kvcache *c, int32_t layer_id, int32_t shared_len,
                            const void *q, void *o, int32_t n_heads, float sm_scale,
                            const pkv_workspace *ws, void *stream);

/*
 * Paged decode through a page table ("KVCache System": the pool is made of
 * pages of page_size consecutive token slots; the 5-D view [n_layers,
 * n_pages, page_size, n_kv_heads, head_dim] is byte-identical to
 * c->k_buffer's [n_layers, size, n_kv_heads, head_dim] with size = n_pages *
 * page_size).  Position j of entry b reads slot
 *   req_to_page[r * max_pages + j / page_size] * page_size + j % page_size,
 * r = c->req_pool_indices[b]; a 16-token stage of the kernel is then a run of
 * consecutive slots.  req_to_page: int32 [c->num_reqs, max_pages] device
 * array (c->num_reqs is its row count); c->req_to_token and c->max_ctx_len
 * are not read.  Otherwise the operation, arguments, results and plan are
 * those of pkv_paged_decode, with c->max_len <= max_pages * page_size.
 * Requires c->size to be a multiple of page_size.  Supported: bf16,
 * head_dim 64 or 128, G and n_kv_heads in {1, 2, 4, 8}.  A page index
 * outside [0, size / page_size) is a device-data error.
 *
 * shared_pages: the caller's statement that the first shared_pages pages of
 * every row of the batch are the same pages (a prefix shared by all
 * requests, "KVCache System" prefix cache hits); 0 states nothing.  It does
 * not change the result: with 8 kv heads, at least 64 shared positions
 * (Ts = shared_pages * page_size), batch >= 2 and room in the workspace it
 * lets the decode read each shared K/V row fewer times than once per
 * request, and merge the two parts; otherwise it is ignored.
 *   - head_dim 128: once per launch.  A tensor-core kernel attends all
 *     batch x G query heads of each kv head to the prefix (read from the
 *     first entry's row) in chunks of at most 512 positions, one CTA per
 *     (chunk, kv head, 256 query rows), while the split kernel takes every
 *     entry's positions past the prefix on the other SMs.  The workspace
 *     then holds (CTAs + batch) x n_heads rows plus ceil(Ts / 512) x batch x
 *     n_heads more, CTAs being the SM count minus the tensor-core kernel's.
 *   - head_dim 64: once per group of 16 / G consecutive requests, inside the
 *     split kernel; the workspace holds (CTAs + batch) x n_heads rows plus
 *     (CTAs + ceil(batch / (16 / G))) x (16 / G) x n_heads more.
 * Every seq_len must be >= Ts; a shorter context, or a row whose leading
 * pages differ from the first entry's (head_dim 128) or its group's
 * (head_dim 64), is a device-data error.  shared_pages < 0, or shared
 * positions beyond c->max_len, returns PKV_ERR_ARG.
 */
int pkv_paged_decode_pages(const pkv_kvcache *c, int32_t layer_id, const int32_t *req_to_page,
                           int32_t max_pages, int32_t page_size, int32_t shared_pages,
                           const void *q, void *o, int32_t n_heads, float sm_scale,
                           const pkv_workspace *ws, void *stream);

/*
 * One decode step of a layer ("Attention Backend": the new tokens' K/V go
 * into the cache, then attention reads it): pkv_kv_write of k_new / v_new
 * (n_new rows at c->out_cache_loc, n_new may be 0) followed by
 * pkv_paged_decode with the automatic plan.  Arguments, layouts, results and
 * errors are those of the two calls made back to back on `stream`; both are
 * validated before either is enqueued.  The tensor-core decode kernel is
 * launched as a programmatic dependent of the write: it reads kv_indptr,
 * req_pool_indices, seq_lens, req_to_token and q while the write runs and
 * waits for the write before reading K/V rows.  Those inputs therefore follow
 * plain stream order (the write never modifies them).  When q (bf16) is in
 * pinned host memory and the workspace has room past the partial rows the
 * call uses, the write also copies q into that room once, and the decode
 * reads the copy after its wait instead of q over the host link; the result
 * is the same either way.
 */
int pkv_decode_step(const pkv_kvcache *c, int32_t layer_id, const void *k_new, const void *v_new,
                    int32_t n_new, const void *q, void *o, int32_t n_heads, float sm_scale,
                    const pkv_workspace *ws, void *stream);

/*
 * pkv_paged_decode with an explicit split size: every entry's context is cut
 * into chunks of `chunk` tokens (a positive multiple of 32; 0 = automatic).
 * The result is the same up to fp32 rounding for any chunk; the workspace
 * must hold ceil(c->max_len / chunk) splits.
 */
int pkv_paged_decode_chunked(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                             int32_t n_heads, float sm_scale, int32_t chunk,
                             const pkv_workspace *ws, void *stream);

/*
 * The plan pkv_paged_decode would use: *chunk tokens per split and
 * *n_splits = ceil(c->max_len / *chunk) splits, or *chunk = 0 and *n_splits =
 * the number of CTAs when the tokens are divided evenly over kv_indptr.
 * Host-only; enqueues nothing.
 */
int pkv_decode_plan(const pkv_kvcache *c, int32_t n_heads, const pkv_workspace *ws,
                    int32_t *chunk, int32_t *n_splits);

/*
 * Ragged paged prefill ("Attention Backend" prefill path).  Entry b has
 * q_len = qo_indptr[b+1] - qo_indptr[b] new tokens (already written to the
 * cache) at the end of a context of kv_len = kv_indptr[b+1] - kv_indptr[b]
 * positions, so its cached prefix is P = kv_len - q_len.  Packed query row
 * p = qo_indptr[b] + i, head h attends over positions j < P + i + 1 when
 * `causal` (the mask of process_attention_mask: a cached prefix is fully
 * visible), else j < kv_len, reading slot req_to_token[req_pool_indices[b], j]
 * of kv head h / G.  q, o: [qo_indptr[batch], n_heads, head_dim] bf16.
 * max_q_len / max_kv_len: host-side upper bounds of q_len and kv_len (grid
 * sizing; max_q_len * G at most 65535 * 256 rows, else PKV_ERR_ARG).  The
 * CTAs launch the kv heads of a query-tile pair together, the pairs of an
 * entry longest first, then the entries.  An entry whose rows [qo_indptr[b], qo_indptr[b+1]) do not lie
 * within [0, qo_indptr[batch]), or whose lengths break these bounds, is a
 * device-data error: its rows of q and o are neither read nor written.
 * `ws` may be NULL.  With a workspace (pkv_workspace_init; its o_part must
 * hold 8 ints per entry) and 2 to 256 entries, a one-CTA planning kernel
 * checks the entries and ranks them by decreasing kv_len into the start of
 * o_part, and the prefill, launched as its programmatic dependent, takes the
 * entries in that order: the longest start first and the short ones fill
 * the SMs at the end.  The result is the same bits in either order.  The
 * workspace serves one call at a time (as for the decode).  Supported: bf16,
 * head_dim 64 or 128 (5th-generation tensor cores, accumulators in tensor
 * memory), G in {1, 2, 4, 8}.
 */
int pkv_paged_prefill(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                      int32_t n_heads, int32_t max_q_len, int32_t max_kv_len, int32_t causal,
                      float sm_scale, const pkv_workspace *ws, void *stream);

/*
 * Paged decode for callers that cannot allocate device memory: code running
 * while another component holds a stream capture open in global mode (where
 * cudaMalloc is not allowed), plugins inside engines whose allocator owns all
 * device memory, or latency-bound loops that cannot take cudaMalloc's
 * implicit synchronisation.  The pages have no counterpart: their decode always
 * receives a workspace.
 *
 * Same operation, arguments and results as pkv_paged_decode, but the split-K
 * partials live in a library-owned device array of 8 MiB (a file-scope
 * __device__ object that every GPU loading the library holds until the
 * process exits).  Nothing is allocated or freed.  The number of splits is
 * capped by what fits in the array for batch x n_heads x head_dim.  When not
 * even one split per (entry, head) fits, contexts of up to 2048 tokens
 * (c->max_len <= 2048) are decoded in one split with o written directly;
 * longer ones, or contexts that would need chunks over 2048 tokens, return
 * PKV_ERR_WORKSPACE.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call on a device shares the one array
 * and leaves its partials there (nothing in it has to start at zero): calls
 * that overlap on the GPU, on any streams, race and give wrong results.
 */
int pkv_paged_decode_noalloc(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                             int32_t n_heads, float sm_scale, void *stream);

/*
 * Synchronise `stream`, then read and clear the calling device's error word.
 * Returns PKV_OK, PKV_ERR_INDEX (an error recorded on the device since the
 * last read) or PKV_ERR_CUDA.  *detail, if non-NULL, receives the first
 * recorded value: the offending slot, page, request row, length or position
 * itself, or one of these codes:
 *   -1000 - k      a decode wait on the copies of stage k gave up;
 *   -2001, -2007   a prefill wait gave up (producer, softmax warps);
 *   -3002 .. -3006 a prefill wait of the thread issuing tensor-core
 *                  instructions gave up;
 *   -100000 - b    a shared prefix was stated, but entry b's leading pages (or
 *                  slots) differ from the first entry's (head_dim 128) or
 *                  from its group's first entry's (head_dim 64);
 *   -200000 - c    shared-prefix CTA c was handed more positions than it
 *                  stages (not expected: the host sizes the grid for it).
 * An offending value can itself be negative (a negative slot, say).
 */
int pkv_last_device_error(void *stream, int64_t *detail);

/* Static, human-readable text for a status code. */
const char *pkv_status_string(int status);

/* Library version string. */
const char *pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
