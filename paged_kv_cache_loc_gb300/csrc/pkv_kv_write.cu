// pkv_kv_write.cu -- K/V cache write k_buffer[layer_id, out_cache_loc] = k
// (AstrAI docs/guides/inference.md, "KVCache System"), and the same write with
// the rotary embedding applied to K first ("KV Cache": RoPE before the write;
// "Rotary Embedding Backend": freqs_cis [max_len, dim/2, 2] cos/sin pairs).
//
// The write is a pure HBM copy: every (token, 16-byte chunk) of the new K and
// V rows is one work item, consecutive threads take consecutive chunks of a
// row, so both the reads of k/v and the scattered row writes are fully
// coalesced 16-byte accesses.  Each thread issues all of its loads before its
// stores to keep several requests in flight.
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// kStep: the write of a decode step (launched with the shared-memory
// carve-out at its maximum, see launch_kv_write); same code otherwise.
template <bool kStep>
__global__ void __launch_bounds__(kThreads) kv_write_kernel(const KvWriteParams p) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int32_t per_buf = static_cast<int32_t>(p.n_new) * p.row_chunks;
    const int32_t total = 2 * per_buf;
    const unsigned kv_blocks = static_cast<unsigned>((total + kThreads * kUnroll - 1) / (kThreads * kUnroll));
    if (blockIdx.x >= kv_blocks) {
        // the CTAs past the rows copy q into the workspace (decode step)
        const int64_t qbase = static_cast<int64_t>(blockIdx.x - kv_blocks) * (kThreads * kUnroll) + threadIdx.x;
        uint4 qv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (qbase + u * kThreads < p.q_chunks) qv[u] = __ldg(static_cast<const uint4 *>(p.q_src) + qbase + u * kThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (qbase + u * kThreads < p.q_chunks) static_cast<uint4 *>(p.q_dst)[qbase + u * kThreads] = qv[u];
        return;
    }
    const int32_t base = blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
    // The row chunk and its slot are independent loads, issued together: the
    // new rows (and slots) may sit in host memory, where each dependent round
    // trip costs microseconds.
    uint4 val[kUnroll];
    long long loc[kUnroll];
    int32_t rem[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int32_t idx = base + u * kThreads;
        rem[u] = -1;
        if (idx < total) {
            const bool is_v = idx >= per_buf;
            rem[u] = is_v ? idx - per_buf : idx;
            loc[u] = __ldg(p.out_cache_loc + rem[u] / p.row_chunks);
            val[u] = __ldg(static_cast<const uint4 *>(is_v ? p.v : p.k) + rem[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        if (rem[u] < 0) continue;
        if (static_cast<unsigned long long>(loc[u]) >= static_cast<unsigned long long>(p.size)) {
            record_error(p.err, loc[u]);
            continue;
        }
        const bool is_v = base + u * kThreads >= per_buf;
        const int32_t c = rem[u] - (rem[u] / p.row_chunks) * p.row_chunks;
        static_cast<uint4 *>(is_v ? p.v_buffer : p.k_buffer)[(p.layer_row0 + loc[u]) * p.row_chunks + c] = val[u];
    }
}

// Rotate the pairs of one 16-byte chunk of a K row.  `pair0` is the index of
// the chunk's first (even, odd) pair within its head; cs points at
// freqs_cis[pos, pair0, 0].
__device__ __forceinline__ uint4 rotate_chunk_bf16(uint4 x, const float *cs) {
    const float4 c0 = *reinterpret_cast<const float4 *>(cs);      // pairs 0,1
    const float4 c1 = *reinterpret_cast<const float4 *>(cs + 4);  // pairs 2,3
    const float cosv[4] = {c0.x, c0.z, c1.x, c1.z};
    const float sinv[4] = {c0.y, c0.w, c1.y, c1.w};
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float re = bf16lo(w[j]), im = bf16hi(w[j]);
        const float ore = re * cosv[j] - im * sinv[j];
        const float oim = re * sinv[j] + im * cosv[j];
        const __nv_bfloat162 r = __floats2bfloat162_rn(ore, oim);
        w[j] = *reinterpret_cast<const uint32_t *>(&r);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 rotate_chunk_f32(uint4 x, const float *cs) {
    const float4 c = *reinterpret_cast<const float4 *>(cs);   // pairs 0,1
    const float re0 = __uint_as_float(x.x), im0 = __uint_as_float(x.y);
    const float re1 = __uint_as_float(x.z), im1 = __uint_as_float(x.w);
    return make_uint4(__float_as_uint(re0 * c.x - im0 * c.y), __float_as_uint(re0 * c.y + im0 * c.x),
                      __float_as_uint(re1 * c.z - im1 * c.w), __float_as_uint(re1 * c.w + im1 * c.z));
}

// The fused write: the first k_blocks CTAs rotate K, one thread per (token,
// chunk offset within a head) for every kv head of the token, so the chunk's
// cos/sin pairs are read once for all heads (a table row would otherwise be
// read once per head) and the heads' K chunks are loads in flight together;
// consecutive threads take consecutive chunks of a head, so each warp's loads
// and stores are whole 256-byte head rows.  The other CTAs copy V like
// kv_write_kernel.  A thread holds kMaxHeads K chunks at a time and takes
// further passes of the head loop for more kv heads: the V-copy CTAs get the
// kernel's register count too, and with 2 chunks a pass (no spills, more CTAs
// per SM) the whole write ran 12 % faster on a 17K-token batch with 8 kv heads
// than with all 8 chunks held at once.
constexpr int kMaxHeads = 2;

template <bool BF16>
__global__ void __launch_bounds__(kThreads) rope_kv_write_kernel(const KvWriteParams p, unsigned k_blocks) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    constexpr int kElemsPerChunk = BF16 ? 8 : 4;
    const int chunks_per_head = p.head_dim / kElemsPerChunk;
    const int n_heads = p.row_chunks / chunks_per_head;
    if (blockIdx.x < k_blocks) {
        const int32_t item = blockIdx.x * kThreads + threadIdx.x;   // (token, chunk offset)
        if (item >= static_cast<int32_t>(p.n_new) * chunks_per_head) return;
        const int32_t i = item / chunks_per_head;
        const int c = item - i * chunks_per_head;
        const long long loc = __ldg(p.out_cache_loc + i);
        const int pos = __ldg(p.positions + i);
        if (static_cast<unsigned long long>(loc) >= static_cast<unsigned long long>(p.size)) {
            record_error(p.err, loc);
            return;
        }
        if (static_cast<unsigned>(pos) >= static_cast<unsigned>(p.max_pos)) {
            record_error(p.err, pos);
            return;
        }
        const uint4 *src = static_cast<const uint4 *>(p.k) + static_cast<int64_t>(i) * p.row_chunks + c;
        uint4 *dst = static_cast<uint4 *>(p.k_buffer) + (p.layer_row0 + loc) * p.row_chunks + c;
        const float *cs = p.freqs_cis + (static_cast<int64_t>(pos) * (p.head_dim / 2) + c * (kElemsPerChunk / 2)) * 2;
        for (int h0 = 0; h0 < n_heads; h0 += kMaxHeads) {
            uint4 x[kMaxHeads];
#pragma unroll
            for (int h = 0; h < kMaxHeads; ++h)
                if (h0 + h < n_heads) x[h] = __ldg(src + (h0 + h) * chunks_per_head);
#pragma unroll
            for (int h = 0; h < kMaxHeads; ++h)
                if (h0 + h < n_heads)
                    dst[(h0 + h) * chunks_per_head] = BF16 ? rotate_chunk_bf16(x[h], cs) : rotate_chunk_f32(x[h], cs);
        }
        return;
    }
    // V: a plain copy
    const int32_t per_buf = static_cast<int32_t>(p.n_new) * p.row_chunks;
    const int32_t base = (blockIdx.x - k_blocks) * (kThreads * kUnroll) + threadIdx.x;
    uint4 val[kUnroll];
    uint4 *dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int32_t idx = base + u * kThreads;
        dst[u] = nullptr;
        if (idx < per_buf) {
            const int32_t i = idx / p.row_chunks;
            const int32_t c = idx - i * p.row_chunks;
            const long long loc = __ldg(p.out_cache_loc + i);
            if (static_cast<unsigned long long>(loc) >= static_cast<unsigned long long>(p.size)) {
                record_error(p.err, loc);
                continue;
            }
            val[u] = __ldg(static_cast<const uint4 *>(p.v) + idx);
            dst[u] = static_cast<uint4 *>(p.v_buffer) + (p.layer_row0 + loc) * p.row_chunks + c;
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
        if (dst[u]) *dst[u] = val[u];
}

inline unsigned grid_for(const KvWriteParams &p) {
    const long long total = 2LL * p.n_new * p.row_chunks;
    return static_cast<unsigned>((total + kThreads * kUnroll - 1) / (kThreads * kUnroll));
}

}  // namespace

cudaError_t launch_kv_write(const KvWriteParams &p, cudaStream_t s, bool step) {
    if (p.n_new == 0) return cudaSuccess;
    if (!step) {
        kv_write_kernel<false><<<grid_for(p), kThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    // The write uses no shared memory.  In a decode step, with the carve-out
    // at its shared maximum, the decode kernel that follows (about 208 KB of
    // shared memory per SM) fits beside it and the SMs need no
    // reconfiguration between the two.  A standalone write keeps the default
    // carve-out of whatever ran before it.
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(kv_write_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const unsigned q_blocks = static_cast<unsigned>((p.q_chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll));
    kv_write_kernel<true><<<grid_for(p) + q_blocks, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rope_kv_write(const KvWriteParams &p, cudaStream_t s) {
    if (p.n_new == 0) return cudaSuccess;
    const long long chunks_per_head = p.head_dim / (p.dtype == PKV_BF16 ? 8 : 4);
    const long long k_items = p.n_new * chunks_per_head;
    const long long v_chunks = p.n_new * p.row_chunks;
    const unsigned k_blocks = static_cast<unsigned>((k_items + kThreads - 1) / kThreads);
    const unsigned v_blocks = static_cast<unsigned>((v_chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll));
    if (p.dtype == PKV_BF16)
        rope_kv_write_kernel<true><<<k_blocks + v_blocks, kThreads, 0, s>>>(p, k_blocks);
    else
        rope_kv_write_kernel<false><<<k_blocks + v_blocks, kThreads, 0, s>>>(p, k_blocks);
    return cudaGetLastError();
}

}  // namespace pkv
