// pkv_decode.cu -- paged decode attention read through req_to_token, split-K
// partials and their merge.
//
// Operation (AstrAI docs/guides/inference.md, "KV Cache" and "Attention
// Backend", decode path with page_size 1): for entry b, query head h,
//   o[b,h] = sum_{j < seq_lens[b]} softmax_j(scale * q[b,h] . K[slot_j, h/G]) V[slot_j, h/G],
//   slot_j = req_to_token[req_pool_indices[b], j].
// The workspace partials follow the pages' decode_o_part / decode_ml_part.
//
// This file holds the CUDA-core split kernel (fp32 storage), the merge
// kernel shared by both dtypes, and the dispatch; bf16 storage runs its split
// pass on tensor cores (pkv_decode_mma.cu).
//
// Design (memory-bound): one CTA per (split, kv head, entry).  Its G query
// heads share every K/V row it reads, so each row leaves HBM once per call.
//   1. the split's int32 slot indices are staged in shared memory once;
//   2. K and V rows (head_dim elements, 128-256 bytes each) are gathered
//      with 16-byte cp.async into a STAGES-deep ring of 32-token tiles;
//   3. each warp owns 8 tokens of a tile and runs its own online softmax:
//      lanes hold head_dim/32 elements of q for all G heads, the per-token
//      partial dots are combined with a reduce-scatter butterfly (one value
//      per lane for G = 4), p goes to warp-private shared memory, and the P.V
//      update has each lane accumulate its head_dim/32 slice for all G heads;
//   4. the 4 warps' (m, l, acc) are combined in shared memory and written as
//      the split's normalised partial (or straight to o when there is one
//      split); a merge kernel rescales and sums the splits.
// Scores live in base-2 units (q is pre-scaled by scale * log2 e).
#include <float.h>

#include <atomic>
#include <type_traits>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kNT = 128;     // threads per CTA
constexpr int kNW = 4;       // warps per CTA
constexpr int kTok = 32;     // tokens per pipeline tile
constexpr int kTPW = kTok / kNW;  // tokens per warp per tile

template <typename T, int D, int G>
struct DecodeCfg {
    static constexpr int kStages = 4;
    static constexpr int kEB = sizeof(T);
    static constexpr int kChunks = D * kEB / 16;           // 16-byte chunks per row
    static constexpr int kEPL = D / 32;                    // elements per lane
    static constexpr int kV = kTPW * G;                    // partial dots per lane per tile
    static constexpr int kLogV = kV == 8 ? 3 : kV == 16 ? 4 : kV == 32 ? 5 : 6;
    static constexpr int kNV = kV >= 32 ? kV / 32 : 1;     // values per lane after reduction
    static constexpr int kRep = kV >= 32 ? 1 : 32 / kV;    // lanes holding the same value
    static constexpr size_t kSlotBytes = kDecodeMaxChunk * 4;
    static constexpr size_t kTileElems = static_cast<size_t>(kTok) * D;
    static constexpr size_t kRingBytes = kStages * 2 * kTileElems * kEB;
    static constexpr size_t kPBytes = kNW * kTPW * G * 4 + kNW * G * 4;
    static constexpr size_t kCombineBytes = (2 * kNW * G + kNW * G * D) * 4;
    static constexpr size_t kSmem =
        kSlotBytes + (kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes) + kPBytes;
    static_assert(kV == 8 || kV == 16 || kV == 32 || kV == 64, "G must be 1, 2, 4 or 8");
    static_assert(kEPL * kEB == 4 || kEPL * kEB == 8 || kEPL * kEB == 16, "lane slice");
};

// Reduce-scatter across the warp: on entry every lane holds V partial values;
// on exit lane l holds in v[0..NV) the warp-wide sums of values
// l*NV .. l*NV+NV-1 (V >= 32) or of value l >> (5 - log2 V) (V < 32).
template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V], int lane) {
    int n = V;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const bool upper = (lane & off) != 0;
            const int half = n / 2;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kNT) decode_split_kernel(const DecodeParams p) {
    using C = DecodeCfg<T, D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    int *slots = reinterpret_cast<int *>(smem);
    T *ring = reinterpret_cast<T *>(smem + C::kSlotBytes);
    const size_t ring_or_combine =
        C::kRingBytes > C::kCombineBytes ? C::kRingBytes : C::kCombineBytes;
    float *pw = reinterpret_cast<float *>(smem + C::kSlotBytes + ring_or_combine);  // [NW][TPW][G]
    float *aw = pw + kNW * kTPW * G;                                                 // [NW][G]

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int r = __ldg(p.req_pool_indices + b);
    if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
        record_error(p.err, r);
        r = 0;
    }
    int n = __ldg(p.seq_lens + b);
    const int n_cap = min(p.max_len, p.max_ctx_len);
    if (n < 0 || n > n_cap) {
        record_error(p.err, n);
        n = max(0, min(n, n_cap));
    }
    const int start = split * p.chunk;
    if (start >= n) {
        if (p.direct && n == 0) {   // single split and empty context: o = 0
            T *o = static_cast<T *>(p.o) + (static_cast<int64_t>(b) * p.n_heads + g * G) * D;
            for (int i = tid; i < G * D; i += kNT) o[i] = Elem<T>::from_f(0.f);
        }
        return;
    }
    const int len = min(p.chunk, n - start);
    const int ntiles = (len + kTok - 1) / kTok;

    // 1. stage the split's slot indices
    const int32_t *row = p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len + start;
    for (int j = tid; j < len; j += kNT) {
        int sl = __ldg(row + j);
        if (static_cast<unsigned long long>(static_cast<long long>(sl)) >=
            static_cast<unsigned long long>(p.size)) {
            record_error(p.err, sl);
            sl = 0;
        }
        slots[j] = sl;
    }

    const int64_t slot_stride = static_cast<int64_t>(p.n_kv_heads) * D;   // elements
    const T *kbase = static_cast<const T *>(p.k_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const T *vbase = static_cast<const T *>(p.v_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;

    // q slice of this lane for the G heads, pre-scaled into base-2 units
    float qf[G][C::kEPL];
    {
        const T *qb = static_cast<const T *>(p.q) +
                      (static_cast<int64_t>(b) * p.n_heads + g * G) * D + lane * C::kEPL;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            load_widen<T, C::kEPL>(qb + h * D, qf[h]);
#pragma unroll
            for (int e = 0; e < C::kEPL; ++e) qf[h][e] *= p.scale_log2;
        }
    }
    __syncthreads();

    auto load_tile = [&](int tile, int buf) {
        T *dk = ring + static_cast<size_t>(buf) * 2 * C::kTileElems;
        T *dv = dk + C::kTileElems;
        const int t0 = tile * kTok;
#pragma unroll
        for (int it = 0; it < (2 * kTok * C::kChunks) / kNT; ++it) {
            const int idx = tid + it * kNT;
            const int is_v = idx / (kTok * C::kChunks);
            const int rem = idx - is_v * (kTok * C::kChunks);
            const int t = rem / C::kChunks;
            const int c = rem - t * C::kChunks;
            const int tok = t0 + t;
            T *dst = (is_v ? dv : dk) + t * D + c * (16 / C::kEB);
            if (tok < len) {
                const T *src = (is_v ? vbase : kbase) + slots[tok] * slot_stride + c * (16 / C::kEB);
                cp_async16(dst, src);
            } else {
                cp_async16(dst, kbase, 0);   // zero fill, nothing read
            }
        }
    };

#pragma unroll
    for (int st = 0; st < C::kStages - 1; ++st) {
        if (st < ntiles) load_tile(st, st);
        cp_async_commit();
    }

    float m_run[C::kNV], l_run[C::kNV];
#pragma unroll
    for (int k = 0; k < C::kNV; ++k) {
        m_run[k] = -INFINITY;
        l_run[k] = 0.f;
    }
    float acc[G][C::kEPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) acc[h][e] = 0.f;

    const bool leader = (lane & (C::kRep - 1)) == 0;

    for (int tile = 0; tile < ntiles; ++tile) {
        cp_async_wait<C::kStages - 2>();
        __syncthreads();
        {
            const int nt = tile + C::kStages - 1;
            if (nt < ntiles) load_tile(nt, nt % C::kStages);
            cp_async_commit();
        }
        const int buf = tile % C::kStages;
        const T *kt = ring + static_cast<size_t>(buf) * 2 * C::kTileElems + warp * kTPW * D;
        const T *vt = kt + C::kTileElems;
        const int valid = min(kTPW, len - tile * kTok - warp * kTPW);
        if (valid <= 0) continue;   // warp-uniform

        // q . k for the warp's 8 tokens and G heads
        float part[C::kV];
#pragma unroll
        for (int t = 0; t < kTPW; ++t) {
            float kf[C::kEPL];
            load_widen<T, C::kEPL>(kt + t * D + lane * C::kEPL, kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < C::kEPL; ++e) a = fmaf(qf[h][e], kf[e], a);
                part[t * G + h] = a;
            }
        }
        warp_reduce_scatter<C::kV>(part, lane);

        // online softmax over the tile, per head
#pragma unroll
        for (int k = 0; k < C::kNV; ++k) {
            const int idx = C::kV >= 32 ? lane * C::kNV + k : (lane >> (5 - C::kLogV));
            const int t = idx / G, h = idx - (idx / G) * G;
            const float s = t < valid ? part[k] : -INFINITY;
            float mx = s;
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[k], mx);
            const float alpha = fast_exp2(m_run[k] - m_new);
            const float pv = fast_exp2(s - m_new);
            float sum = pv;
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l_run[k] = l_run[k] * alpha + sum;
            m_run[k] = m_new;
            if (leader) {
                pw[(warp * kTPW + t) * G + h] = pv;
                if (t == 0) aw[warp * G + h] = alpha;
            }
        }
        __syncwarp();

        // acc = alpha * acc + sum_t p_t v_t
        {
            float al[G];
#pragma unroll
            for (int h = 0; h < G; ++h) al[h] = aw[warp * G + h];
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < C::kEPL; ++e) acc[h][e] *= al[h];
#pragma unroll
            for (int t = 0; t < kTPW; ++t) {
                float vf[C::kEPL];
                load_widen<T, C::kEPL>(vt + t * D + lane * C::kEPL, vf);
                const float *pt = pw + (warp * kTPW + t) * G;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float ph = pt[h];
#pragma unroll
                    for (int e = 0; e < C::kEPL; ++e) acc[h][e] = fmaf(ph, vf[e], acc[h][e]);
                }
            }
        }
        __syncwarp();
    }

    // 4. combine the warps
    cp_async_wait<0>();
    __syncthreads();
    float *red_m = reinterpret_cast<float *>(ring);   // [NW][G]
    float *red_l = red_m + kNW * G;                  // [NW][G]
    float *red_acc = red_l + kNW * G;                // [NW][G][D]
#pragma unroll
    for (int k = 0; k < C::kNV; ++k) {
        const int idx = C::kV >= 32 ? lane * C::kNV + k : (lane >> (5 - C::kLogV));
        const int t = idx / G, h = idx - (idx / G) * G;
        if (leader && t == 0) {
            red_m[warp * G + h] = m_run[k];
            red_l[warp * G + h] = l_run[k];
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) red_acc[(warp * G + h) * D + lane * C::kEPL + e] = acc[h][e];
    __syncthreads();

    const int64_t bh0 = static_cast<int64_t>(b) * p.n_heads + g * G;
    for (int i = tid; i < G * D; i += kNT) {
        const int h = i / D, e = i - (i / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNW; ++w) M = fmaxf(M, red_m[w * G + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            const float sc = fast_exp2(red_m[w * G + h] - M);
            L += red_l[w * G + h] * sc;
            O += red_acc[(w * G + h) * D + e] * sc;
        }
        const float out = O / L;
        if (p.direct) {
            static_cast<T *>(p.o)[(bh0 + h) * D + e] = Elem<T>::from_f(out);
        } else {
            const int64_t ps = (bh0 + h) * p.n_splits + split;
            p.o_part[ps * D + e] = out;
            if (e == 0) {
                p.ml_part[ps * 2] = M;
                p.ml_part[ps * 2 + 1] = L;
            }
        }
    }
}

// Merge: o = sum_s l_s 2^(m_s - M) o_s / sum_s l_s 2^(m_s - M) over the
// entry's non-empty splits.  One CTA per (entry, head); 4 groups of D/4
// threads, each group sums every 4th split with float4 loads.
template <typename T, int D>
__global__ void __launch_bounds__(kNT) decode_merge_kernel(const DecodeParams p) {
    constexpr int kCols = D / 4;            // float4 columns
    constexpr int kGroups = kNT / kCols;    // 4 (D=128) or 8 (D=64)
    __shared__ float wts[kDecodeMaxSplits];
    __shared__ float red[kNT / 32];
    __shared__ float4 part[kGroups][kCols];

    const int bh = blockIdx.x;
    const int b = bh / p.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_cap = min(p.max_len, p.max_ctx_len);
    const int n = max(0, min(__ldg(p.seq_lens + b), n_cap));
    const int nv = (n + p.chunk - 1) / p.chunk;
    T *out = static_cast<T *>(p.o) + static_cast<int64_t>(bh) * D;
    if (nv == 0) {
        for (int e = tid; e < D; e += kNT) out[e] = Elem<T>::from_f(0.f);
        return;
    }
    const float *ml = p.ml_part + static_cast<int64_t>(bh) * p.n_splits * 2;
    const float *op = p.o_part + static_cast<int64_t>(bh) * p.n_splits * D;

    float mx = -INFINITY;
    for (int s = tid; s < nv; s += kNT) mx = fmaxf(mx, ml[2 * s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int w = 1; w < kNT / 32; ++w) M = fmaxf(M, red[w]);
    __syncthreads();

    float sum = 0.f;
    for (int s = tid; s < nv; s += kNT) {
        const float w = ml[2 * s + 1] * fast_exp2(ml[2 * s] - M);
        wts[s] = w;
        sum += w;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kNT / 32; ++w) L += red[w];

    const int col = tid % kCols, grp = tid / kCols;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = grp; s < nv; s += kGroups) {
        const float w = wts[s];
        const float4 x = *reinterpret_cast<const float4 *>(op + static_cast<int64_t>(s) * D + col * 4);
        a.x = fmaf(w, x.x, a.x);
        a.y = fmaf(w, x.y, a.y);
        a.z = fmaf(w, x.z, a.z);
        a.w = fmaf(w, x.w, a.w);
    }
    part[grp][col] = a;
    __syncthreads();
    if (grp == 0) {
        float4 t = part[0][col];
#pragma unroll
        for (int q = 1; q < kGroups; ++q) {
            t.x += part[q][col].x;
            t.y += part[q][col].y;
            t.z += part[q][col].z;
            t.w += part[q][col].w;
        }
        const float inv = 1.f / L;
        out[col * 4 + 0] = Elem<T>::from_f(t.x * inv);
        out[col * 4 + 1] = Elem<T>::from_f(t.y * inv);
        out[col * 4 + 2] = Elem<T>::from_f(t.z * inv);
        out[col * 4 + 3] = Elem<T>::from_f(t.w * inv);
    }
}

template <typename T, int D, int G>
cudaError_t run(const DecodeParams &p, cudaStream_t s) {
    using C = DecodeCfg<T, D, G>;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        // bf16: the split pass runs on tensor cores
        cudaError_t e = launch_decode_split_mma(p, D, G, s);
        if (e != cudaSuccess) return e;
        if (p.balanced) return launch_decode_merge_balanced(p, D, s);
        if (p.direct) return cudaSuccess;
        decode_merge_kernel<T, D><<<p.batch * p.n_heads, kNT, 0, s>>>(p);
        return cudaGetLastError();
    } else {
    static std::atomic<uint64_t> attr_done{0};   // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(decode_split_kernel<T, D, G>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    dim3 grid(p.n_splits, p.n_kv_heads, p.batch);
    decode_split_kernel<T, D, G><<<grid, kNT, C::kSmem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.direct) return e;
    decode_merge_kernel<T, D><<<p.batch * p.n_heads, kNT, 0, s>>>(p);
    return cudaGetLastError();
    }
}

template <typename T, int D>
cudaError_t run_group(const DecodeParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run<T, D, 1>(p, s);
        case 2: return run<T, D, 2>(p, s);
        case 4: return run<T, D, 4>(p, s);
        case 8: return run<T, D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool decode_supported(int dtype, int head_dim, int group) {
    return (dtype == PKV_F32 || dtype == PKV_BF16) && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode(const DecodeParams &p, int dtype, int head_dim, int group,
                          cudaStream_t s) {
    if (!decode_supported(dtype, head_dim, group)) return cudaErrorNotSupported;
    if (p.batch == 0) return cudaSuccess;
    if (dtype == PKV_BF16)
        return head_dim == 128 ? run_group<__nv_bfloat16, 128>(p, group, s)
                               : run_group<__nv_bfloat16, 64>(p, group, s);
    return head_dim == 128 ? run_group<float, 128>(p, group, s) : run_group<float, 64>(p, group, s);
}

}  // namespace pkv
