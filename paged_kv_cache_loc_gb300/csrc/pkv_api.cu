// pkv_api.cu -- the C ABI declared in include/pkv.h: host-side argument
// checks, the decode split plan, workspace bookkeeping, the per-device error
// word, and dispatch to the kernels.  Nothing here allocates device memory.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <initializer_list>
#include <mutex>

#include "pkv.h"
#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace {

// The per-device error word written by the kernels (see pkv_common.cuh).
__device__ pkv::DevErr g_err;

constexpr uint32_t kWsMagic = 0x706b7731u;   // "pkw1"
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    pkv::DevErr *err = nullptr;
    int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Device-side address of g_err and the SM count of the current device,
// looked up once per device with that device current.
int device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.err) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_err) != cudaSuccess) return PKV_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_ERR_CUDA;
        d.err = static_cast<pkv::DevErr *>(ptr);
        d.sms = sms;
    }
    *out = d;
    return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Memory the kernels may dereference: device or managed memory, or
// registered (pinned) host memory mapped at the same address, which the GPU
// reads and writes over the host link.  Anything else (an unregistered host
// address, say) is refused before launching, since touching it would fault
// the device.  Null entries are optional arguments the caller checked.
bool device_visible(const void *p) {
    if (!p) return true;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // not sticky: clear it
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}
// Registered host memory (the kernels reach it over the host link).
bool host_memory(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}
int check_visible(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (!device_visible(p)) return PKV_ERR_ARG;
    return PKV_OK;
}

int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

int map_launch(cudaError_t e) {
    if (e == cudaSuccess) return PKV_OK;
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    return PKV_ERR_CUDA;
}

// Checks shared by every entry point that touches the pool.
int check_pool(const pkv_kvcache *c, int32_t layer_id) {
    if (!c || !c->k_buffer || !c->v_buffer) return PKV_ERR_ARG;
    if (c->dtype != PKV_F32 && c->dtype != PKV_BF16) return PKV_ERR_ARG;
    if (c->n_layers <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->size <= 0)
        return PKV_ERR_ARG;
    if (c->size > INT32_MAX) return PKV_ERR_ARG;   // slots are int32
    if (layer_id < 0 || layer_id >= c->n_layers) return PKV_ERR_ARG;
    if (!aligned16(c->k_buffer) || !aligned16(c->v_buffer)) return PKV_ERR_ARG;
    const int64_t row_bytes = static_cast<int64_t>(c->n_kv_heads) * c->head_dim * elem_bytes(c->dtype);
    if (row_bytes % 16) return PKV_ERR_ARG;
    return PKV_OK;
}

// Checks for the attention entry points (req_to_token indirection).
int check_attn(const pkv_kvcache *c, int32_t n_heads, const void *q, const void *o) {
    if (!c->req_to_token || !c->req_pool_indices) return PKV_ERR_ARG;
    if (c->num_reqs <= 0 || c->max_ctx_len <= 0 || c->batch < 0 || c->max_len < 0) return PKV_ERR_ARG;
    if (c->max_len > c->max_ctx_len) return PKV_ERR_ARG;
    if (n_heads <= 0 || n_heads % c->n_kv_heads) return PKV_ERR_ARG;
    if (c->batch > 0 && (!q || !o || !aligned16(q) || !aligned16(o))) return PKV_ERR_ARG;
    if (c->batch > 65535) return PKV_ERR_ARG;   // grid z
    return PKV_OK;
}

int ws_check(const pkv_workspace *ws) {
    if (!ws || ws->magic != kWsMagic || !ws->base) return PKV_ERR_WORKSPACE;
    return PKV_OK;
}

// The decode work plan.
//  balanced: chosen when the caller asked for the automatic plan, passed
//    kv_indptr, the shape has a balanced kernel and the workspace holds
//    (n_parts + batch) * n_heads partial rows.  n_parts CTAs (one per SM, or
//    fewer: when the batch holds less than ~32 tokens per SM, and in the two
//    cases below) share all tokens of the batch equally.
//  chunked: each entry's context is cut into chunks; about four CTAs per SM
//    if every context were max_len long, 64..2048 tokens in steps of 32, never
//    more splits than the workspace holds (one split without a workspace).
struct Plan {
    int balanced = 0;
    int32_t chunk = 0;
    int32_t n_splits = 1;
    int32_t n_parts = 0;
};

bool ws_holds(const pkv_workspace *ws, int64_t rows, int head_dim) {
    const int64_t cap_o =
        static_cast<int64_t>(ws->max_batch) * ws->n_heads * ws->max_splits * ws->head_dim;
    const int64_t cap_ml = static_cast<int64_t>(ws->max_batch) * ws->n_heads * ws->max_splits * 2;
    return rows * head_dim <= cap_o && rows * 2 <= cap_ml;
}

int make_plan(const pkv_kvcache *c, int32_t n_heads, int sms, const pkv_workspace *ws,
              int32_t chunk_req, Plan *out) {
    const int64_t max_len = c->max_len > 0 ? c->max_len : 1;
    const int64_t batch = c->batch > 0 ? c->batch : 1;
    const int group = n_heads / c->n_kv_heads;
    const bool have_ws = ws_check(ws) == PKV_OK;
    if (chunk_req == 0 && c->kv_indptr && have_ws &&
        pkv::decode_balanced_supported(c->dtype, c->head_dim, group, c->n_kv_heads)) {
        int64_t parts = (max_len * batch + 31) / 32;   // at least ~32 tokens (2 stages) per CTA
        int64_t cap = sms > 0 ? sms : 1;
        // One request with 96 to 320 positions per SM: 4/5 of the SMs, each
        // CTA then streaming a longer piece.  Measured on GB300 (152 SMs), B=1
        // at 16K / 32K positions: 23.8-25.2 / 35.2-35.6 us against 26.0-26.2
        // / 35.6-36.0 us on every SM.  Shorter contexts (4K: two 16-token
        // stages per CTA) and batched decodes measured fastest as before.
        if (batch == 1 && max_len >= 96 * cap && max_len < 320 * cap) cap = cap * 4 / 5;
        // A batch of fewer than 1024 positions per SM: 12/13 of the SMs (140
        // of 152).  With every SM streaming, some SMs of a GB300 read 10-15 %
        // slower than the rest (the same ones every call, set by the chip's
        // layout), and a short call waits for them; with a few SMs idle the
        // rest read evenly.  Measured on two GB300s, 32 requests x 77.7K
        // tokens: 62.5 / 61.2 us against 65.0 / 62.5 us on every SM.  Calls
        // of several thousand positions per SM need every SM's bandwidth
        // (2 GB: 330 us on 152 CTAs, 353 on 140).
        else if (batch > 1 && max_len * batch < 1024 * cap) cap = cap * 12 / 13;
        if (parts > cap) parts = cap;
        if (parts < 1) parts = 1;
        if (ws_holds(ws, (parts + batch) * n_heads, c->head_dim)) {
            out->balanced = 1;
            out->n_parts = static_cast<int32_t>(parts);
            out->chunk = 0;
            out->n_splits = static_cast<int32_t>(parts);
            return PKV_OK;
        }
    }
    int64_t chunk = chunk_req;
    if (chunk == 0) {
        const int64_t units = batch * c->n_kv_heads;
        const int64_t target = static_cast<int64_t>(sms > 0 ? sms : 1) * 4;
        chunk = (max_len * units + target - 1) / target;
        chunk = (chunk + 31) / 32 * 32;
        if (chunk < 64) chunk = 64;
        if (chunk > pkv::kDecodeMaxChunk) chunk = pkv::kDecodeMaxChunk;
        const int64_t cap_splits =
            have_ws ? (ws->max_splits < pkv::kDecodeMaxSplits ? ws->max_splits : pkv::kDecodeMaxSplits)
                    : 1;
        if ((max_len + chunk - 1) / chunk > cap_splits) {
            chunk = (max_len + cap_splits - 1) / cap_splits;
            chunk = (chunk + 31) / 32 * 32;
        }
        if (chunk > pkv::kDecodeMaxChunk) return PKV_ERR_WORKSPACE;
    }
    if (chunk <= 0 || chunk % 32 || chunk > pkv::kDecodeMaxChunk) return PKV_ERR_ARG;
    const int64_t n_splits = (max_len + chunk - 1) / chunk;
    if (n_splits > pkv::kDecodeMaxSplits) return PKV_ERR_ARG;
    out->balanced = 0;
    out->chunk = static_cast<int32_t>(chunk);
    out->n_splits = static_cast<int32_t>(n_splits);
    out->n_parts = 0;
    return PKV_OK;
}

// Validates a decode call and fills its kernel parameters; *empty is set when
// there is nothing to launch (batch 0).  Enqueues nothing.
int decode_prepare(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                   int32_t n_heads, float sm_scale, int32_t chunk, const pkv_workspace *ws,
                   pkv::DecodeParams *out, bool *empty) {
    *empty = false;
    int rc = check_pool(c, layer_id);
    if (rc) return rc;
    rc = check_attn(c, n_heads, q, o);
    if (rc) return rc;
    if (!c->seq_lens) return PKV_ERR_ARG;
    if (!isfinite(sm_scale)) return PKV_ERR_ARG;
    const int group = n_heads / c->n_kv_heads;
    if (!pkv::decode_supported(c->dtype, c->head_dim, group)) return PKV_ERR_UNSUPPORTED;
    if (c->batch == 0) {
        *empty = true;
        return PKV_OK;
    }
    if (q == o) return PKV_ERR_ARG;
    DeviceInfo di;
    rc = device_info(&di);
    if (rc) return rc;
    rc = check_visible({c->k_buffer, c->v_buffer, c->req_to_token, c->req_pool_indices, c->seq_lens,
                        c->kv_indptr, q, o, ws ? ws->base : nullptr});
    if (rc) return rc;
    Plan plan;
    rc = make_plan(c, n_heads, di.sms, ws, chunk, &plan);
    if (rc) return rc;

    pkv::DecodeParams &p = *out;
    p = pkv::DecodeParams{};
    p.balanced = plan.balanced;
    p.n_parts = plan.n_parts;
    p.kv_indptr = c->kv_indptr;
    p.direct = !plan.balanced && plan.n_splits == 1;
    if (!p.direct) {
        rc = ws_check(ws);
        if (rc) return rc;
        const int64_t rows = plan.balanced
                                 ? (static_cast<int64_t>(plan.n_parts) + c->batch) * n_heads
                                 : static_cast<int64_t>(c->batch) * n_heads * plan.n_splits;
        if (!ws_holds(ws, rows, c->head_dim)) return PKV_ERR_WORKSPACE;
        p.o_part = ws->o_part;
        p.ml_part = ws->ml_part;
    }
    p.q = q;
    p.o = o;
    p.k_buffer = c->k_buffer;
    p.v_buffer = c->v_buffer;
    p.req_to_token = c->req_to_token;
    p.req_pool_indices = c->req_pool_indices;
    p.seq_lens = c->seq_lens;
    p.size = c->size;
    p.layer_row0 = static_cast<int64_t>(layer_id) * c->size;
    p.n_kv_heads = c->n_kv_heads;
    p.n_heads = n_heads;
    p.num_reqs = c->num_reqs;
    p.max_ctx_len = c->max_ctx_len;
    p.batch = c->batch;
    p.max_len = c->max_len;
    p.chunk = plan.chunk;
    p.n_splits = plan.n_splits;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.err = di.err;
    return PKV_OK;
}

int decode_impl(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o, int32_t n_heads,
                float sm_scale, int32_t chunk, const pkv_workspace *ws, void *stream) {
    pkv::DecodeParams p;
    bool empty = false;
    int rc = decode_prepare(c, layer_id, q, o, n_heads, sm_scale, chunk, ws, &p, &empty);
    if (rc || empty) return rc;
    return map_launch(pkv::launch_decode(p, c->dtype, c->head_dim, p.n_heads / p.n_kv_heads,
                                         static_cast<cudaStream_t>(stream)));
}

// Validates a cache write and fills its kernel parameters; *empty is set
// when there is nothing to launch (n_new 0).  Enqueues nothing.
int kv_write_prepare(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                     int32_t n_new, const float *freqs_cis, int32_t max_pos,
                     const int32_t *positions, bool rope, pkv::KvWriteParams *out, bool *empty) {
    *empty = false;
    int rc = check_pool(c, layer_id);
    if (rc) return rc;
    if (n_new < 0) return PKV_ERR_ARG;
    if (n_new == 0) {
        *empty = true;
        return PKV_OK;
    }
    if (!k || !v || !c->out_cache_loc || !aligned16(k) || !aligned16(v)) return PKV_ERR_ARG;
    const int64_t row_chunks =
        static_cast<int64_t>(c->n_kv_heads) * c->head_dim * elem_bytes(c->dtype) / 16;
    if (2 * static_cast<int64_t>(n_new) * row_chunks >= INT32_MAX) return PKV_ERR_ARG;
    if (rope) {
        if (!freqs_cis || !positions || max_pos <= 0 || !aligned16(freqs_cis)) return PKV_ERR_ARG;
        if ((c->head_dim * elem_bytes(c->dtype)) % 16) return PKV_ERR_ARG;   // chunks stay in a head
    }
    DeviceInfo di;
    rc = device_info(&di);
    if (rc) return rc;
    rc = check_visible({c->k_buffer, c->v_buffer, c->out_cache_loc, k, v, rope ? freqs_cis : nullptr,
                        rope ? positions : nullptr});
    if (rc) return rc;
    pkv::KvWriteParams &p = *out;
    p = pkv::KvWriteParams{};
    p.k = k;
    p.v = v;
    p.k_buffer = c->k_buffer;
    p.v_buffer = c->v_buffer;
    p.out_cache_loc = c->out_cache_loc;
    p.n_new = n_new;
    p.size = c->size;
    p.layer_row0 = static_cast<int64_t>(layer_id) * c->size;
    p.row_chunks = static_cast<int32_t>(row_chunks);
    p.head_dim = c->head_dim;
    p.dtype = c->dtype;
    p.freqs_cis = freqs_cis;
    p.positions = positions;
    p.max_pos = max_pos;
    p.err = di.err;
    return PKV_OK;
}

int kv_write_impl(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                  int32_t n_new, const float *freqs_cis, int32_t max_pos,
                  const int32_t *positions, bool rope, void *stream) {
    pkv::KvWriteParams p;
    bool empty = false;
    int rc = kv_write_prepare(c, layer_id, k, v, n_new, freqs_cis, max_pos, positions, rope, &p,
                              &empty);
    if (rc || empty) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return map_launch(rope ? pkv::launch_rope_kv_write(p, s) : pkv::launch_kv_write(p, s));
}

}  // namespace

extern "C" {

size_t pkv_workspace_bytes(int32_t max_batch, int32_t n_heads, int32_t head_dim,
                           int32_t max_splits) {
    if (max_batch < 1 || n_heads < 1 || head_dim < 1 || max_splits < 1) return 0;
    const size_t units = static_cast<size_t>(max_batch) * n_heads * max_splits;
    const size_t o_bytes = (units * head_dim * sizeof(float) + 255) / 256 * 256;
    return o_bytes + units * 2 * sizeof(float);
}

int pkv_workspace_init(void *base, size_t bytes, int32_t max_batch, int32_t n_heads,
                       int32_t head_dim, int32_t max_splits, pkv_workspace *out) {
    if (!out || !base || (reinterpret_cast<uintptr_t>(base) & 255u)) return PKV_ERR_ARG;
    const size_t need = pkv_workspace_bytes(max_batch, n_heads, head_dim, max_splits);
    if (need == 0) return PKV_ERR_ARG;
    if (bytes < need) return PKV_ERR_WORKSPACE;
    const size_t units = static_cast<size_t>(max_batch) * n_heads * max_splits;
    const size_t o_bytes = (units * head_dim * sizeof(float) + 255) / 256 * 256;
    out->base = base;
    out->bytes = bytes;
    out->max_batch = max_batch;
    out->n_heads = n_heads;
    out->head_dim = head_dim;
    out->max_splits = max_splits;
    out->o_part = static_cast<float *>(base);
    out->ml_part = reinterpret_cast<float *>(static_cast<char *>(base) + o_bytes);
    out->magic = kWsMagic;
    return PKV_OK;
}

int pkv_kv_write(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                 int32_t n_new, void *stream) {
    return kv_write_impl(c, layer_id, k, v, n_new, nullptr, 0, nullptr, false, stream);
}

int pkv_rope_kv_write(const pkv_kvcache *c, int32_t layer_id, const void *k, const void *v,
                      int32_t n_new, const float *freqs_cis, int32_t max_pos,
                      const int32_t *positions, void *stream) {
    return kv_write_impl(c, layer_id, k, v, n_new, freqs_cis, max_pos, positions, true, stream);
}

int pkv_paged_decode(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                     int32_t n_heads, float sm_scale, const pkv_workspace *ws, void *stream) {
    return decode_impl(c, layer_id, q, o, n_heads, sm_scale, 0, ws, stream);
}

// Shared-prefix mode, when it applies and fits; otherwise p is left as it is
// (the plain balanced decode).  Its partials follow the private rows in the
// workspace.
//  - head_dim 128: the prefix is read once per launch, by a tensor-core
//    kernel over all batch x G query rows of each kv head (256 rows per CTA),
//    the prefix cut into chunks of at most kGroupChunk positions; the private
//    role takes the SMs that kernel leaves free.
//  - head_dim 64: the group role runs inside the split kernel, one warp per
//    kv head, at most 1024 group positions per CTA, with at least one CTA
//    left for the private role; the prefix is read once per group of 16 / G
//    requests.
// Prefix positions per group-role CTA: four 128-key tiles.  On the
// prefix-shared workload (64 requests, 2048 shared positions, 8 kv heads) that
// is 32 group CTAs, which end before the private role on the other 120 SMs.
constexpr int64_t kGroupChunk = 512;

void use_shared_prefix(const pkv_kvcache *c, int32_t n_heads, int64_t shared_len,
                       const pkv_workspace *ws, pkv::DecodeParams *p) {
    const int group = n_heads / c->n_kv_heads;
    if (shared_len < 64 || c->batch < 2 || c->n_kv_heads != 8 || !p->balanced ||
        shared_len * c->batch > INT32_MAX)
        return;
    if (c->head_dim == 128) {
        DeviceInfo di;
        if (device_info(&di) != PKV_OK) return;
        const int64_t row_blocks = (static_cast<int64_t>(c->batch) * group + pkv::kGroupRows - 1) /
                                   pkv::kGroupRows;
        int64_t chunks = (shared_len + kGroupChunk - 1) / kGroupChunk;
        const int64_t chunk_len = ((shared_len + chunks - 1) / chunks + 127) / 128 * 128;
        chunks = (shared_len + chunk_len - 1) / chunk_len;
        const int64_t group_ctas = chunks * c->n_kv_heads * row_blocks;
        int64_t parts = di.sms - group_ctas;
        if (parts > p->n_parts) parts = p->n_parts;
        if (parts < 1) parts = 1;
        const int64_t unit0 = (parts + c->batch) * n_heads;
        if (row_blocks > 65535 || !ws_holds(ws, unit0 + chunks * c->batch * n_heads, c->head_dim))
            return;
        p->n_parts = static_cast<int32_t>(parts);
        p->n_splits = static_cast<int32_t>(parts);
        p->shared_len = static_cast<int32_t>(shared_len);
        p->group_tc = 1;
        p->group_chunks = static_cast<int32_t>(chunks);
        p->group_chunk_len = static_cast<int32_t>(chunk_len);
        p->group_reqs = 1;
        p->n_groups = static_cast<int32_t>(c->batch);
        p->group_unit0 = unit0;
        return;
    }
    const int64_t reqs = 16 / group;
    const int64_t n_groups = (c->batch + reqs - 1) / reqs;
    const int64_t min_group_ctas = (n_groups * shared_len + 1023) / 1024;
    const int64_t unit0 = (static_cast<int64_t>(p->n_parts) + c->batch) * n_heads;
    const int64_t units = unit0 + (p->n_parts + n_groups) * reqs * n_heads;
    if (p->n_parts < min_group_ctas + 1 || !ws_holds(ws, units, c->head_dim)) return;
    p->shared_len = static_cast<int32_t>(shared_len);
    p->group_reqs = static_cast<int32_t>(reqs);
    p->n_groups = static_cast<int32_t>(n_groups);
    p->group_unit0 = unit0;
}

int pkv_paged_decode_shared(const pkv_kvcache *c, int32_t layer_id, int32_t shared_len,
                            const void *q, void *o, int32_t n_heads, float sm_scale,
                            const pkv_workspace *ws, void *stream) {
    if (!c) return PKV_ERR_ARG;
    if (shared_len < 0 || (c->batch > 0 && shared_len > c->max_len)) return PKV_ERR_ARG;
    pkv::DecodeParams p;
    bool empty = false;
    int rc = decode_prepare(c, layer_id, q, o, n_heads, sm_scale, 0, ws, &p, &empty);
    if (rc || empty) return rc;
    use_shared_prefix(c, n_heads, shared_len, ws, &p);
    return map_launch(pkv::launch_decode(p, c->dtype, c->head_dim, n_heads / c->n_kv_heads,
                                         static_cast<cudaStream_t>(stream)));
}

int pkv_paged_decode_pages(const pkv_kvcache *c, int32_t layer_id, const int32_t *req_to_page,
                           int32_t max_pages, int32_t page_size, int32_t shared_pages,
                           const void *q, void *o, int32_t n_heads, float sm_scale,
                           const pkv_workspace *ws, void *stream) {
    if (!c || !req_to_page || max_pages <= 0 || page_size <= 0) return PKV_ERR_ARG;
    if (c->size <= 0 || c->size % page_size) return PKV_ERR_ARG;
    if (static_cast<int64_t>(max_pages) * page_size > INT32_MAX) return PKV_ERR_ARG;
    const int64_t shared_len = static_cast<int64_t>(shared_pages) * page_size;
    if (shared_pages < 0 || (c->batch > 0 && shared_len > c->max_len)) return PKV_ERR_ARG;
    // the cache as the decode sees it: positions reach max_pages * page_size
    // and request rows index the page table; req_to_token is not read
    pkv_kvcache cc = *c;
    cc.req_to_token = req_to_page;
    cc.max_ctx_len = max_pages * page_size;
    pkv::DecodeParams p;
    bool empty = false;
    int rc = decode_prepare(&cc, layer_id, q, o, n_heads, sm_scale, 0, ws, &p, &empty);
    if (rc || empty) return rc;
    if (!pkv::decode_balanced_supported(c->dtype, c->head_dim, n_heads / c->n_kv_heads, c->n_kv_heads))
        return PKV_ERR_UNSUPPORTED;
    p.req_to_token = nullptr;
    p.req_to_page = req_to_page;
    p.max_pages = max_pages;
    p.page_size = page_size;
    p.n_pages = c->size / page_size;
    use_shared_prefix(c, n_heads, shared_len, ws, &p);
    return map_launch(pkv::launch_decode(p, c->dtype, c->head_dim, n_heads / c->n_kv_heads,
                                         static_cast<cudaStream_t>(stream)));
}

int pkv_decode_step(const pkv_kvcache *c, int32_t layer_id, const void *k_new, const void *v_new,
                    int32_t n_new, const void *q, void *o, int32_t n_heads, float sm_scale,
                    const pkv_workspace *ws, void *stream) {
    // both calls are validated before either is enqueued
    pkv::KvWriteParams wp;
    bool no_write = false;
    int rc = kv_write_prepare(c, layer_id, k_new, v_new, n_new, nullptr, 0, nullptr, false, &wp,
                              &no_write);
    if (rc) return rc;
    pkv::DecodeParams dp;
    bool no_decode = false;
    rc = decode_prepare(c, layer_id, q, o, n_heads, sm_scale, 0, ws, &dp, &no_decode);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the tensor-core split kernels read metadata and q before waiting on
    // the write; the others are launched in plain stream order
    dp.pdl = !no_write && !no_decode &&
             pkv::decode_balanced_supported(c->dtype, c->head_dim, n_heads / c->n_kv_heads, c->n_kv_heads);
    // q in host memory: every CTA holding a piece of an entry would read the
    // entry's q over the host link.  When the workspace has room past the
    // partial rows this call uses, the write's extra CTAs copy q there once,
    // and the decode reads that copy after its wait for the write.
    if (dp.pdl && dp.balanced && c->dtype == PKV_BF16 && host_memory(q)) {
        const int64_t rows = (static_cast<int64_t>(dp.n_parts) + c->batch) * n_heads;
        const int64_t cap = static_cast<int64_t>(ws->max_batch) * ws->n_heads * ws->max_splits * ws->head_dim * 4;
        const int64_t off = (rows * c->head_dim * 4 + 255) / 256 * 256;
        const int64_t qbytes = static_cast<int64_t>(c->batch) * n_heads * c->head_dim * 2;
        if (off + qbytes <= cap) {
            wp.q_src = q;
            wp.q_dst = reinterpret_cast<char *>(ws->o_part) + off;
            wp.q_chunks = qbytes / 16;
            dp.q = wp.q_dst;
            dp.q_staged = 1;
        }
    }
    if (!no_write) {
        rc = map_launch(pkv::launch_kv_write(wp, s, true));
        if (rc) return rc;
    }
    if (no_decode) return PKV_OK;
    return map_launch(pkv::launch_decode(dp, c->dtype, c->head_dim, n_heads / c->n_kv_heads, s));
}

int pkv_paged_decode_chunked(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                             int32_t n_heads, float sm_scale, int32_t chunk,
                             const pkv_workspace *ws, void *stream) {
    if (chunk < 0) return PKV_ERR_ARG;
    return decode_impl(c, layer_id, q, o, n_heads, sm_scale, chunk, ws, stream);
}

int pkv_decode_plan(const pkv_kvcache *c, int32_t n_heads, const pkv_workspace *ws,
                    int32_t *chunk, int32_t *n_splits) {
    if (!c || !chunk || !n_splits || c->n_kv_heads <= 0 || n_heads <= 0 || c->max_len < 0 ||
        n_heads % c->n_kv_heads)
        return PKV_ERR_ARG;
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    Plan plan;
    rc = make_plan(c, n_heads, di.sms, ws, 0, &plan);
    if (rc) return rc;
    *chunk = plan.chunk;
    *n_splits = plan.n_splits;
    return PKV_OK;
}

int pkv_paged_prefill(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                      int32_t n_heads, int32_t max_q_len, int32_t max_kv_len, int32_t causal,
                      float sm_scale, const pkv_workspace *ws, void *stream) {
    int rc = check_pool(c, layer_id);
    if (rc) return rc;
    rc = check_attn(c, n_heads, q, o);
    if (rc) return rc;
    if (!c->qo_indptr || !c->kv_indptr) return PKV_ERR_ARG;
    if (max_q_len < 0 || max_kv_len < 0 || max_q_len > max_kv_len || max_kv_len > c->max_ctx_len)
        return PKV_ERR_ARG;
    if (!isfinite(sm_scale)) return PKV_ERR_ARG;
    const int group = n_heads / c->n_kv_heads;
    if (!pkv::prefill_supported(c->dtype, c->head_dim, group)) return PKV_ERR_UNSUPPORTED;
    if (c->batch == 0 || max_q_len == 0) return PKV_OK;
    if (q == o) return PKV_ERR_ARG;
    if (static_cast<int64_t>(max_q_len) * group / 64 + 1 > INT32_MAX) return PKV_ERR_ARG;
    if ((static_cast<int64_t>(max_q_len) * group + 255) / 256 > 65535) return PKV_ERR_ARG;   // grid y: query-tile pairs
    DeviceInfo di;
    rc = device_info(&di);
    if (rc) return rc;
    if (ws) {
        rc = ws_check(ws);
        if (rc) return rc;
    }
    rc = check_visible({c->k_buffer, c->v_buffer, c->req_to_token, c->req_pool_indices, c->qo_indptr,
                        c->kv_indptr, q, o, ws ? ws->base : nullptr});
    if (rc) return rc;
    pkv::PrefillParams p{};
    p.q = q;
    p.o = o;
    p.k_buffer = c->k_buffer;
    p.v_buffer = c->v_buffer;
    p.req_to_token = c->req_to_token;
    p.req_pool_indices = c->req_pool_indices;
    p.qo_indptr = c->qo_indptr;
    p.kv_indptr = c->kv_indptr;
    p.size = c->size;
    p.layer_row0 = static_cast<int64_t>(layer_id) * c->size;
    p.n_kv_heads = c->n_kv_heads;
    p.n_heads = n_heads;
    p.num_reqs = c->num_reqs;
    p.max_ctx_len = c->max_ctx_len;
    p.batch = c->batch;
    p.causal = causal ? 1 : 0;
    p.max_q_len = max_q_len;
    p.max_kv_len = max_kv_len;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.err = di.err;
    if (ws) {   // room for the entry order: 8 ints per entry at the start of o_part
        const int64_t cap = static_cast<int64_t>(ws->max_batch) * ws->n_heads * ws->max_splits * ws->head_dim;
        if (8LL * c->batch <= cap) p.plan = reinterpret_cast<int32_t *>(ws->o_part);
    }
    return map_launch(pkv::launch_prefill(p, c->dtype, c->head_dim, group,
                                          static_cast<cudaStream_t>(stream)));
}

int pkv_last_device_error(void *stream, int64_t *detail) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    pkv::DevErr host{};
    if (cudaMemcpy(&host, di.err, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (!host.flag) return PKV_OK;
    if (detail) *detail = host.detail;
    if (cudaMemset(di.err, 0, sizeof host) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_ERR_INDEX;
}

const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported variant (dtype, head_dim or group size)";
        case PKV_ERR_WORKSPACE: return "workspace missing, uninitialised or too small";
        case PKV_ERR_INDEX: return "device data out of range (slot, request row or length)";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

const char *pkv_version(void) { return "pkv 0.1.0 (sm_103a)"; }

}  // extern "C"
