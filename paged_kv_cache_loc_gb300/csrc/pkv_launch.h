// pkv_launch.h -- internal launch interfaces between the C ABI (pkv_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct DevErr;

// K/V cache write (optionally with the rotary embedding applied to K).
struct KvWriteParams {
    const void *k;              // [n_new, n_kv_heads, head_dim]
    const void *v;
    void *k_buffer;             // pool base
    void *v_buffer;
    const int32_t *out_cache_loc;
    int64_t n_new;
    int64_t size;               // slots per layer
    int64_t layer_row0;         // layer_id * size
    int32_t row_chunks;         // 16-byte chunks per (layer, slot) row
    int32_t head_dim;
    int32_t dtype;              // pkv_dtype
    const float *freqs_cis;     // rope only: [max_pos, head_dim/2, 2]
    const int32_t *positions;   // rope only: [n_new]
    int32_t max_pos;
    DevErr *err;
    // decode step only: copy q_chunks 16-byte chunks from q_src to q_dst (q
    // moved from host memory into the workspace once, for the decode)
    const void *q_src;
    void *q_dst;
    int64_t q_chunks;
};

// Split-K paged decode.
struct DecodeParams {
    const void *q;              // [batch, n_heads, head_dim]
    void *o;                    // [batch, n_heads, head_dim]
    const void *k_buffer;
    const void *v_buffer;
    const int32_t *req_to_token;
    const int32_t *req_pool_indices;
    const int32_t *seq_lens;
    float *o_part;              // [batch, n_heads, n_splits, head_dim]
    float *ml_part;             // [batch, n_heads, n_splits, 2]
    int64_t size;
    int64_t layer_row0;
    int32_t n_kv_heads;
    int32_t n_heads;
    int32_t num_reqs;
    int32_t max_ctx_len;
    int32_t batch;
    int32_t max_len;
    int32_t chunk;              // tokens per split (multiple of 32)
    int32_t n_splits;           // ceil(max_len / chunk)
    int32_t direct;             // 1: single split, write o directly (no merge)
    float scale_log2;           // sm_scale * log2(e)
    DevErr *err;
    // Balanced mode: the split grid is n_parts CTAs that share the flattened
    // token space [0, kv_indptr[batch]) equally; CTA c's piece of entry b is
    // partial row (c + b) of o_part / ml_part ([n_parts + batch, n_heads, ...]).
    const int32_t *kv_indptr;
    int32_t balanced;
    int32_t n_parts;
    // 1: the split kernel is launched as a programmatic dependent of the
    // cache write before it; it reads metadata, slot indices and q at once
    // and waits (griddepcontrol.wait) before its first K/V row read.
    int32_t pdl;
    // 1 (with pdl): q is a copy the cache write makes in the workspace, so it
    // is read only after the wait.
    int32_t q_staged;
    // Page-table addressing (page_size > 0): position j of request row r is
    // slot req_to_page[r * max_pages + j / page_size] * page_size +
    // j % page_size, with pages < n_pages; req_to_token is not read.
    const int32_t *req_to_page;
    int32_t max_pages;
    int32_t page_size;
    int64_t n_pages;
    // Shared prefix (balanced mode, 8 kv heads): positions [0, shared_len)
    // of every entry map to the same slots.  The first CTAs of the grid
    // (the group role) stream that prefix once per group of group_reqs
    // consecutive entries, the requests' heads side by side as the score
    // block's 16 columns; the others (the private role) take the balanced
    // partition of the positions [shared_len, seq_len) of all entries.  The
    // group role's piece of group gi in its CTA cs is written for member u,
    // head h to unit group_unit0 + ((cs + gi) * group_reqs + u) * n_heads + h
    // of o_part / ml_part.  shared_len 0: off.
    int32_t shared_len;
    int32_t group_reqs;
    int32_t n_groups;
    int64_t group_unit0;
    // Shared prefix read once per launch (bf16, head_dim 128): the group role
    // is a separate tensor-core kernel (launch_shared_group_tc) over all
    // batch x G query rows of each kv head, one CTA per (prefix chunk of
    // group_chunk_len positions, kv head, 256 query rows); its partial of
    // chunk k for entry b, head h is unit group_unit0 + (k * batch + b) *
    // n_heads + h.  All n_parts CTAs of the split kernel take the private
    // role.  The group kernel is launched as a programmatic dependent of the
    // split kernel, on the SMs the split leaves free, and waits for it
    // (griddepcontrol.wait) only before it exits; the merge, launched as the
    // group kernel's dependent, then sees both.
    int32_t group_tc;
    int32_t group_chunks;
    int32_t group_chunk_len;
};

// Ragged causal prefill.
struct PrefillParams {
    const void *q;              // [total_q, n_heads, head_dim]
    void *o;
    const void *k_buffer;
    const void *v_buffer;
    const int32_t *req_to_token;
    const int32_t *req_pool_indices;
    const int32_t *qo_indptr;
    const int32_t *kv_indptr;
    int64_t size;
    int64_t layer_row0;
    int32_t n_kv_heads;
    int32_t n_heads;
    int32_t num_reqs;
    int32_t max_ctx_len;
    int32_t batch;
    int32_t causal;
    int32_t max_q_len;
    int32_t max_kv_len;
    float scale_log2;
    DevErr *err;
    // With a workspace: 8 ints per entry rank (entry, request row, first
    // packed row, q_len, kv_len, valid, 0, 0), the entries by decreasing
    // kv_len, written by the plan kernel that runs first; CTA z takes rank z.
    int32_t *plan;
    // Shared-prefix group role (launch_shared_group_tc), not used by the
    // prefill: rows are the batch x G (entry, head) pairs of q [batch,
    // n_heads, head_dim]; the keys are positions [0, shared_len) of the
    // first entry's row (req_to_token, or the page table when page_size >
    // 0), chunk_len of them per CTA; each CTA writes fp32 partials (o / l,
    // then (m, l)) for its rows to o_part / ml_part at unit0 + (chunk *
    // batch + b) * n_heads + h.
    const int32_t *req_to_page;
    int32_t max_pages;
    int32_t page_size;
    int64_t n_pages;
    int32_t shared_len;
    int32_t chunk_len;
    float *o_part;
    float *ml_part;
    int64_t unit0;
};

constexpr int kDecodeMaxChunk = 2048;   // slot indices staged per split (or per piece)
constexpr int kDecodeMaxSplits = 1024;  // merge kernel limit
constexpr int kPlanMaxBatch = 256;      // prefill entries ordered by the plan kernel (one CTA)

// Each returns cudaSuccess or the launch error.  Unsupported variants return
// cudaErrorNotSupported and enqueue nothing.
// step: the write of pkv_decode_step (see pkv_kv_write.cu)
cudaError_t launch_kv_write(const KvWriteParams &p, cudaStream_t s, bool step = false);
cudaError_t launch_rope_kv_write(const KvWriteParams &p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams &p, int dtype, int head_dim, int group,
                          cudaStream_t s);
bool decode_supported(int dtype, int head_dim, int group);
// bf16 split pass on tensor cores (pkv_decode_mma.cu); the merge is launched
// by launch_decode.
cudaError_t launch_decode_split_mma(const DecodeParams &p, int head_dim, int group,
                                    cudaStream_t s);
// Whether the bf16 balanced mode is available for this shape.
bool decode_balanced_supported(int dtype, int head_dim, int group, int n_kv_heads);
// Merge of the balanced mode (pkv_decode_mma.cu).
cudaError_t launch_decode_merge_balanced(const DecodeParams &p, int head_dim, cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams &p, int dtype, int head_dim, int group,
                           cudaStream_t s);
// The prefill runs on tcgen05 with accumulators in TMEM for bf16 head_dim 64
// and 128 (pkv_prefill_tc.cu).
bool prefill_supported(int dtype, int head_dim, int group);
// The shared-prefix group role of a decode with p.group_tc set
// (pkv_prefill_tc.cu); launched before the split kernel.
cudaError_t launch_shared_group_tc(const DecodeParams &p, int group, cudaStream_t s);
constexpr int kGroupRows = 256;          // query rows per group-role CTA (two 128-row tiles)

}  // namespace pkv
